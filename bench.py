#!/usr/bin/env python
"""Benchmark of the radix-cache attention hot path on one GB300 (or N replicas).

One step = the whole agent-loop workload through librx: 40 calls sharing a
3,000-token preamble with U[150, 250]-token suffixes, extend batches chosen by
the in-batch prefix rule, 64 decode steps over all 40 calls, finish.  Every
step starts from an empty cache, so it repeats the same cache decisions: match,
lock, allocate, req_to_token upload, kv_store, extend attention, decode plan,
shared-prefix + private decode attention with log-sum-exp merge, insert,
unlock.  Q/K/V are seeded synthetic bf16 N(0, 1) values resident in HBM before
the timed region (``value``); ``e2e`` repeats the step with the inputs in pinned
host memory, copied to the device inside the timed region, and the attention
outputs read back.

Prints one JSON line.  ``--impl reference`` times the CPU oracle instead.
"""

import os

for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse  # noqa: E402
import json  # noqa: E402
import statistics  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import tempfile  # noqa: E402
import time  # noqa: E402

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "extend query-tok/s and decode attn GB/s (% of GB300 HBM peak) on radix KV pool"
L2_FLUSH_BYTES = 256 << 20
L2_BYTES = 126 << 20            # GB300 L2 capacity


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="agent_loop")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    return ap.parse_args()


# DRAM bytes (read + write) per launch of the dominant kernel, from the ncu
# captures summarised in profiles/ (cold L2, the current kernels):
# decode_fused_kernel on one agent_loop and one long_shared decode step; the
# extend kernel averaged over the launches of one step (long_shared: 2,
# fork_tree: 130), as `achieved` averages over them.  None (absent) where no
# capture of that launch exists.
TRAFFIC = {
    ("agent_loop", "rx_decode_attention"): 44.534e6 + 0.006e6,
    ("long_shared", "rx_decode_attention"): 406.35e6 + 16.01e6,
    ("long_shared", "rx_extend_attention"): (2230.64e6 + 3158.90e6) / 2,
    ("fork_tree", "rx_extend_attention"): (5711.18e6 + 887.04e6) / 130,
}


def max_over_ranks(x, world, device):
    """The largest of every rank's x (time of a step: the job is as slow as
    its slowest replica); x itself on one rank."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank, seconds, world):
    """Whole-job throughput of `world` replicas that each process
    units_per_rank units in the (max over ranks) time `seconds`."""
    return world * units_per_rank / seconds


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d["hbm_gbs"], d["bf16_tflops"], "measured"
    return 6800.0, 1900.0, "fallback"


# ------------------------------------------------------------------ clocks
class Clocks:
    """nvidia-smi sampling of SM clock and throttle reasons in the background."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(index)], stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        self.t0 = None
        self.t1 = None

    def begin(self):
        self.t0 = time.time()

    def end(self):
        self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        with open(self.file.name) as f:
            lines = [ln.strip() for ln in f if ln.strip()]
        os.unlink(self.file.name)
        import datetime
        rows = []
        for ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
            except ValueError:
                continue
        # samples inside the timed region (all samples if the region was too short)
        inside = [r for r in rows if self.t0 is not None and self.t1 is not None
                  and self.t0 - 0.15 <= r[0] <= self.t1 + 0.15]
        use = inside if inside else rows
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for _, clk, cmax, flags in use:
            sm.append(clk)
            mx.append(cmax)
            for n, v in zip(names, flags):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm),
                "samples_in_timed_region": len(inside)}


# --------------------------------------------------------------- CPU oracle
def oracle_rate(wl, rows_of, budget_s=12.0, seed=0):
    """Oracle throughput (query tokens/s) on a bounded sample.

    Bookkeeping of the whole workload is run in full; attention is computed
    in fp64 for a random sample of the workload's queries (extend tokens and
    decode tokens) until ``budget_s`` is spent, and the per-query cost is
    scaled to the whole workload."""
    from oracle import attention as oatt
    from oracle.harness import run_bookkeeping

    t0 = time.perf_counter()
    trace, _ = run_bookkeeping(wl.oracle_waves(), wl.num_slots, wl.decode_steps)
    t_book = time.perf_counter() - t0
    n_ext = trace.prefilled
    n_dec = sum(len(w) for w in wl.waves) * wl.decode_steps
    queries = []
    for b in trace.batches:
        for rid, m, row in b:
            for i in range(m, len(row)):
                queries.append(("e", rid, m, i))
    rng = np.random.default_rng(seed)
    order = rng.permutation(len(queries))
    dec_q = [(r.rid, t) for w in wl.waves for r in w for t in range(wl.decode_steps)]
    dorder = rng.permutation(len(dec_q))
    done = 0
    t_att = 0.0
    k = 0
    while t_att < budget_s and k < len(order):
        # alternate extend and decode queries in proportion to the workload
        if dec_q and rng.random() < n_dec / (n_ext + n_dec):
            rid, t = dec_q[dorder[k % len(dorder)]]
            r = wl.requests[rid]
            ctx = np.concatenate([wl.prompt_store_index(r), wl.output_store_index(r)[:t + 1]])
            q, kk, vv = rows_of("q", [wl.output_store_index(r)[t]]), rows_of("k", ctx), rows_of("v", ctx)
            s0 = time.perf_counter()
            oatt.decode_attention(q[0], kk, vv)
        else:
            _, rid, m, i = queries[order[k]]
            r = wl.requests[rid]
            pidx = wl.prompt_store_index(r)
            q, kk, vv = rows_of("q", [pidx[i]]), rows_of("k", pidx[:i + 1]), rows_of("v", pidx[:i + 1])
            s0 = time.perf_counter()
            oatt.softmax_attention(q, kk, vv, [i + 1])
        t_att += time.perf_counter() - s0
        done += 1
        k += 1
    total_q = n_ext + n_dec
    est = t_book + t_att * total_q / max(1, done)
    return {
        "value": total_q / est,
        "unit": "query-tok/s",
        "cores": 1,
        "kind": "oracle",
        "sample": (f"bookkeeping of the whole workload ({t_book:.2f} s) + fp64 attention of "
                   f"{done} randomly drawn queries of {total_q} ({t_att:.1f} s), scaled to all "
                   "queries; numpy single-threaded"),
        "seconds": t_book + t_att,
    }


def run_reference(args, rank, world):
    if rank != 0:
        return
    from radix_tree_prefix_gb300 import workloads
    wl = workloads.WORKLOADS[args.workload]()
    import torch

    def make_rows():
        g = workloads.make_values(wl, "cpu")

        def rows_of(kind, idx):
            t = torch.from_numpy(np.asarray(idx, dtype=np.int64))
            return g[kind][0].index_select(0, t).double().numpy()
        return rows_of

    rows_of = make_rows()
    oracle_rate(wl, rows_of, budget_s=1.0)      # warm-up (imports, caches)
    vals = []
    t0 = time.perf_counter()
    for s in range(args.steps):
        r = oracle_rate(wl, rows_of, budget_s=max(1.0, 60.0 / max(1, args.steps)), seed=s)
        vals.append(r["value"])
    wall = time.perf_counter() - t0
    value = statistics.mean(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "query-tok/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * wall / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, **{k: v for k, v in wl.describe().items()
                                            if k != "workload"}},
        "cpu_baseline": {"value": value, "unit": "query-tok/s", "cores": 1, "kind": "oracle",
                         "sample": r["sample"]},
        "e2e": {"value": value, "unit": "query-tok/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU arm
def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    import torch
    import torch.distributed as dist

    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import __graft_entry__
    __graft_entry__.build()
    from radix_tree_prefix_gb300 import rx, workloads
    from radix_tree_prefix_gb300.engine import Engine, GatherInputs, PreparedInputs

    wl = workloads.WORKLOADS[args.workload]()
    layers = list(range(wl.num_layers))
    values = workloads.make_values(wl, dev, layers)
    prepared = PreparedInputs(GatherInputs(wl, values, layers))
    eng = Engine(wl, device=dev, inputs=prepared, layers=layers)
    trace = eng.run()                       # records the inputs of every batch/step
    prepared.freeze()
    torch.cuda.synchronize()
    rx.device_check()
    n_ext = trace.prefilled
    n_dec = sum(len(w) for w in wl.waves) * wl.decode_steps
    q_per_step = n_ext + n_dec
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    clocks = Clocks(local)          # started before warm-up: its start-up is not timed
    for _ in range(args.warmup):
        eng.run()
    torch.cuda.synchronize()
    time.sleep(0.3)

    # ---------------- timed: inputs resident in HBM
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    eng.timing = True
    eng.kernel_events = []
    launches0 = eng.gpu_launches
    step_ev = []
    stream = torch.cuda.current_stream()
    clocks.begin()
    wall0 = time.perf_counter()
    for _ in range(args.steps):
        flush.zero_()                                   # L2 flushed between steps
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        t = eng.run()
        e1.record(stream)
        step_ev.append((e0, e1))
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    clocks.end()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    launches = eng.gpu_launches - launches0
    assert t.as_tuple() == trace.as_tuple(), "timed steps made different cache decisions"
    rx.device_check()
    step_ms = [a.elapsed_time(b) for a, b in step_ev]
    ms = max_over_ranks(sum(step_ms) / len(step_ms), world, dev)
    value = job_rate(q_per_step, ms / 1000.0, world)

    kinds = {}
    for kind, a, b, work in eng.kernel_events:
        d = kinds.setdefault(kind, {"ms": 0.0, "launches": 0, "work": 0.0})
        d["ms"] += a.elapsed_time(b)
        d["launches"] += 1
        d["work"] += work
    hbm_peak, bf16_peak, peak_src = peaks()
    ext = kinds.get("extend", {"ms": 0.0, "launches": 0, "work": 0.0})
    dec = kinds.get("decode", {"ms": 0.0, "launches": 0, "work": 0.0})
    ext_tflops = ext["work"] / (ext["ms"] / 1e3) / 1e12 if ext["ms"] else 0.0
    dec_gbs = dec["work"] / (dec["ms"] / 1e3) / 1e9 if dec["ms"] else 0.0
    extend_info = {
        "qtok_s": n_ext * args.steps / (ext["ms"] / 1e3) if ext["ms"] else None,
        "tflops": ext_tflops, "frac_of_bf16_peak": ext_tflops / bf16_peak,
        "ms_per_step": ext["ms"] / args.steps, "launches_per_step": ext["launches"] / args.steps,
        "flop_per_step": ext["work"] / args.steps}
    n_dec_launches = args.steps * len(wl.waves) * wl.decode_steps * len(layers)
    decode_info = {
        "gbs": dec_gbs, "frac_of_hbm_peak": dec_gbs / hbm_peak,
        "ms_per_step": dec["ms"] / args.steps, "launches_per_step": dec["launches"] / args.steps,
        "bytes_per_step": dec["work"] / args.steps,
        "note": ("decode working set fits in L2; L2 is flushed between steps only, so "
                 "later decode steps of a step read KV that is partly L2-resident (effective GB/s)")
        if dec["launches"] and dec["work"] / max(1, n_dec_launches) < L2_BYTES else None}
    if ext["ms"] >= dec["ms"]:
        roof = {"kernel": "rx_extend_attention", "bound": "tensor", "achieved": ext_tflops,
                "peak": bf16_peak, "unit": "TFLOP/s", "frac": ext_tflops / bf16_peak,
                "traffic": TRAFFIC.get((args.workload, "rx_extend_attention")),
                "peak_source": f"{peak_src} bf16_tflops (burst)"}
    else:
        roof = {"kernel": "rx_decode_attention", "bound": "hbm", "achieved": dec_gbs,
                "peak": hbm_peak, "unit": "GB/s", "frac": dec_gbs / hbm_peak,
                "traffic": TRAFFIC.get((args.workload, "rx_decode_attention")),
                "peak_source": f"{peak_src} hbm_gbs"}

    # ---------------- e2e: host inputs copied in, outputs read back
    e2e = None
    if not args.no_e2e:
        host_inputs = PreparedInputs(prepared.source, host=True)
        host_inputs.ext = dict(prepared.ext)
        host_inputs.dec = dict(prepared.dec)
        host_inputs.order = list(prepared.order)
        host_inputs.freeze()
        d2h = {"bytes": 0}
        # pinned host buffers for the outputs, allocated in the untimed first
        # run and reused in call order (each step ends with a synchronize)
        sinks = []
        sink_i = [0]

        # outputs go back on a side stream once they are written, while the
        # main stream runs on
        out_stream = torch.cuda.Stream(dev)
        main_stream = torch.cuda.current_stream(dev)

        def grab(outs):
            ready = torch.cuda.Event()
            ready.record(main_stream)
            out_stream.wait_event(ready)
            for o, lse in outs.values():
                for x in (o, lse):
                    x.record_stream(out_stream)
                    i = sink_i[0]
                    if i == len(sinks) or sinks[i].shape != x.shape:
                        h = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
                        if i == len(sinks):
                            sinks.append(h)
                        else:
                            sinks[i] = h
                    with torch.cuda.stream(out_stream):
                        sinks[i].copy_(x, non_blocking=True)
                    sink_i[0] = i + 1
                    d2h["bytes"] += x.numel() * x.element_size()

        # output tensors reused run to run (each run ends with a synchronize,
        # so the previous run's reads of them are done)
        eng2 = Engine(wl, device=dev, inputs=host_inputs, layers=layers,
                      on_extend=lambda b, r, p, q, outs: grab(outs),
                      on_decode_wave=lambda s, r, c, outs, i: grab(outs), reuse_outputs=True)
        eng2.run()
        torch.cuda.synchronize()
        sink_i[0] = 0
        host_inputs.h2d_bytes = 0
        d2h["bytes"] = 0
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            flush.zero_()
            eng2.run()
            torch.cuda.synchronize()
            sink_i[0] = 0
        e2e_s = max_over_ranks((time.perf_counter() - t0) / args.steps, world, dev)
        e2e = {"value": job_rate(q_per_step, e2e_s, world), "unit": "query-tok/s",
               "h2d_bytes_per_step": host_inputs.h2d_bytes // args.steps,
               "d2h_bytes_per_step": d2h["bytes"] // args.steps,
               "ms_per_step": e2e_s * 1e3}

    cpu = None
    if rank == 0 and not args.no_cpu and world == 1:
        def rows_of(kind, idx):
            t = torch.from_numpy(np.asarray(idx, dtype=np.int64)).to(dev)
            return values[kind][0].index_select(0, t).double().cpu().numpy()
        cpu = oracle_rate(wl, rows_of)
        cpu.pop("seconds", None)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "query-tok/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": wl.name, **{k: v for k, v in wl.describe().items()
                                                if k != "workload"},
                       "query_tokens_per_step": q_per_step, "extend_query_tokens": n_ext,
                       "decode_query_tokens": n_dec,
                       "l2": "flushed between timed steps (256 MiB write, outside the step events)",
                       "parallelism": "replicas" if world > 1 else "single",
                       "wall_s_timed_region_incl_flush": wall},
            "extend": extend_info, "decode": decode_info, "roofline": roof,
            "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches, "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

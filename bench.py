#!/usr/bin/env python
"""Benchmark of the radix-cache attention hot path on one GB300 (or N replicas).

One step = the whole multi-turn chat workload through librx: 256 sessions x 8
turns over a shared 2,000-token system prompt, each turn 200 new user tokens
and 32 decoded tokens, 16 full-attention layers, 16 query / 4 KV heads,
head_dim 256 (64 KiB of KV per token).  Every step starts from an empty cache,
so it repeats the same cache decisions: match, lock, allocate, req_to_token
upload, kv_store, extend attention, decode plan, shared-prefix + private
decode attention with log-sum-exp merge, insert, unlock.  Q/K/V are seeded
synthetic bf16 N(0, 1) values resident in HBM before the timed region
(``value``); ``e2e`` repeats the step with the inputs in page-locked host
memory, copied to the device inside the timed region, and every attention
output read back to the host through a bounded ring of buffers.  The same line
carries, per other workload (agent loop, long shared prefix, fork tree), its
step time and the extend, decode and kv_store rates (``configs``).

Prints one JSON line.  ``--impl reference`` times the CPU oracle instead;
``--only kv_store`` times the kv_store kernel alone at the shape of the
workload's largest extend batch (a small case for profiler captures).
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
DEFAULT_WORKLOAD = "multi_turn_chat"
# other workloads measured in the same run, each with its own object in the line
SIDE_WORKLOADS = ("agent_loop", "long_shared", "fork_tree")
SIDE_STEPS = 10                 # timed steps of each side workload (3 warm-up)
E2E_RING_BYTES = 24 << 30       # device (and page-locked host) bytes of the e2e output ring
E2E_INPUT_RING = 4              # e2e input buffers (positions in flight: 3)


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="leave out the other workloads' objects")
    ap.add_argument("--only", choices=["kv_store"], default=None)
    return ap.parse_args(argv)


# DRAM bytes (read + write) per launch of the dominant kernel, from the ncu
# captures summarised in profiles/ (cold L2, the current kernels):
# decode_fused_kernel on one agent_loop and one long_shared decode step; the
# extend kernel per launch (one launch per wave and layer, as `achieved`
# averages over launches); multi_turn_chat's decode
# launch scaled from a capture of one multi_turn_chat_small decode launch by
# the ratio of algorithmic bytes (the full workload's pool is beyond the
# capture size rule).  None (absent) where no capture of that launch exists.
TRAFFIC = {
    ("agent_loop", "rx_decode_attention"): 44.534e6 + 0.006e6,
    ("long_shared", "rx_decode_attention"): 406.35e6 + 16.01e6,
    # one launch per wave: long_shared's two batches (captured as two
    # launches before they were launched together), summed
    ("long_shared", "rx_extend_attention"): 2230.64e6 + 3158.90e6,
    # one wave's launch (26 batches), from its capture
    ("fork_tree", "rx_extend_attention"): 983.37e6 + 1269.09e6,
    # (69.452 MB read + 0.609 MB written) / 69.865 MB algorithmic on the
    # multi_turn_chat_small launch, times the full workload's 1.0940 GB of
    # algorithmic bytes per decode launch
    ("multi_turn_chat", "rx_decode_attention"): (69.452e6 + 0.609e6) / 69.865e6 * 1.0940e9,
}


def config_of(wl, world):
    """The workload's description as both arms print it (identical keys)."""
    return {"workload": wl.name, **{k: v for k, v in wl.describe().items() if k != "workload"},
            "l2": "inputs larger than L2, and L2 flushed between timed steps (256 MiB write, "
                  "outside the step events)",
            "parallelism": (f"{world} replicas, subtree-affine shards (no collective in the "
                            "data path)") if world > 1 else "single"}


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


def job_rate(units_per_rank, seconds, world, device=None):
    """Whole-job throughput of `world` replicas: the units all ranks
    processed (each rank its own share) in the (max over ranks) time
    `seconds`."""
    if world <= 1:
        return units_per_rank / seconds
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(units_per_rank)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item()) / seconds


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
        self.result = None

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
def _pairs(trace, wl):
    """Visible (query, key) pairs of one layer: extend query i of a prompt
    sees keys 0..i; decode step t of a request sees its prompt and t + 1
    decode tokens."""
    ext = 0
    for b in trace.batches:
        for rid, m, row in b:
            n = len(row)
            ext += (n * (n + 1) - m * (m + 1)) // 2
    dec = 0
    T = wl.decode_steps
    for w in wl.waves:
        for r in w:
            p = len(wl.prompt_tokens(r))
            dec += T * p + T * (T + 1) // 2
    return ext, dec


def oracle_bookkeeping(wl):
    """The oracle's request flow over the whole workload, timed."""
    from oracle.harness import run_bookkeeping
    t0 = time.perf_counter()
    trace, _ = run_bookkeeping(wl.oracle_waves(), wl.num_slots, wl.decode_steps,
                                   page_size=wl.page_size)
    return trace, time.perf_counter() - t0


def oracle_rate(wl, budget_s=12.0, seed=0, booked=None, n_requests=8):
    """Oracle throughput (query tokens/s) from a bounded sample.

    The oracle's bookkeeping runs over the whole workload (or ``booked`` =
    (trace, seconds) of such a run is reused).  Attention is computed in fp64
    at one layer with all heads for the queries of ``n_requests`` seeded
    requests (extend and decode queries, in random order) until ``budget_s``
    is spent; its time per visible (query, key) pair is scaled to every pair
    of every layer of the workload.  The oracle's time does not depend on the
    values, so they are seeded normal draws made here."""
    from oracle import attention as oatt

    trace, t_book = booked if booked is not None else oracle_bookkeeping(wl)
    n_ext = trace.prefilled
    n_dec = sum(len(w) for w in wl.waves) * wl.decode_steps
    ext_pairs, dec_pairs = _pairs(trace, wl)
    rng = np.random.default_rng(seed)
    rids = sorted(wl.requests)
    pick = set(int(x) for x in rng.choice(rids, size=min(n_requests, len(rids)), replace=False))
    queries = []
    for b in trace.batches:
        for rid, m, row in b:
            if rid in pick:
                queries += [i + 1 for i in range(m, len(row))]
    for rid in pick:
        p = len(wl.prompt_tokens(wl.requests[rid]))
        queries += [p + t + 1 for t in range(wl.decode_steps)]
    queries = [queries[i] for i in rng.permutation(len(queries))]
    ctx = max(queries)
    k = rng.standard_normal((ctx, wl.num_kv_heads, wl.head_dim))
    v = rng.standard_normal((ctx, wl.num_kv_heads, wl.head_dim))
    q = rng.standard_normal((1, wl.num_q_heads, wl.head_dim))
    done = pairs = 0
    t_att = 0.0
    for n in queries:
        if t_att >= budget_s:
            break
        s0 = time.perf_counter()
        oatt.softmax_attention(q, k[:n], v[:n], [n])
        t_att += time.perf_counter() - s0
        done += 1
        pairs += n
    total_q = n_ext + n_dec
    est = t_book + t_att / max(1, pairs) * (ext_pairs + dec_pairs) * wl.num_layers
    return {
        "value": total_q / est,
        "unit": "query-tok/s",
        "cores": 1,
        "host_cpus": os.cpu_count(),
        "blas_threads": int(os.environ.get("OPENBLAS_NUM_THREADS", "1")),
        "kind": "oracle",
        "sample": (f"bookkeeping of the whole workload ({t_book:.2f} s) + fp64 attention, layer "
                   f"0, all {wl.num_q_heads} heads, of {done} queries drawn from {len(pick)} "
                   f"seeded requests ({t_att:.1f} s, {pairs} of the layer's "
                   f"{ext_pairs + dec_pairs} visible query-key pairs), scaled by pairs to all "
                   f"{wl.num_layers} layers and {total_q} queries; numpy single-threaded"),
        "seconds": t_book + t_att,
    }


def run_reference(args, rank, world):
    """The oracle timed as it stands on one host core: its bookkeeping of the
    whole workload once (before the warm-up steps), then per step a bounded
    attention sample (oracle_rate); value = mean over the timed steps."""
    if rank != 0:
        return
    from radix_tree_prefix_gb300 import workloads
    wl = workloads.WORKLOADS[args.workload]()
    booked = oracle_bookkeeping(wl)
    per_step = max(0.5, 60.0 / max(1, args.steps))
    for s in range(args.warmup):
        oracle_rate(wl, budget_s=min(1.0, per_step), seed=1000 + s, booked=booked)
    vals = []
    t0 = time.perf_counter()
    for s in range(args.steps):
        r = oracle_rate(wl, budget_s=per_step, seed=s, booked=booked)
        vals.append(r["value"])
    wall = time.perf_counter() - t0
    value = statistics.mean(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "query-tok/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * wall / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(wl, world),
        "cpu_baseline": {"value": value, "unit": "query-tok/s", "cores": 1,
                         "host_cpus": r["host_cpus"], "blas_threads": r["blas_threads"],
                         "kind": "oracle", "sample": r["sample"] + f"; mean of {args.steps} steps"},
        "e2e": {"value": value, "unit": "query-tok/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU arm
def _kind_stats(events, steps):
    kinds = {}
    for kind, a, b, work in events:
        d = kinds.setdefault(kind, {"ms": 0.0, "launches": 0, "work": 0.0})
        d["ms"] += a.elapsed_time(b)
        d["launches"] += 1
        d["work"] += work
    for d in kinds.values():
        d["steps"] = steps
    return kinds


def _rates(kinds, n_ext, hbm_peak, bf16_peak, steps, n_dec_launch_bytes=None):
    zero = {"ms": 0.0, "launches": 0, "work": 0.0}
    ext, dec, st = (kinds.get(k, zero) for k in ("extend", "decode", "kv_store"))
    ext_tflops = ext["work"] / (ext["ms"] / 1e3) / 1e12 if ext["ms"] else 0.0
    dec_gbs = dec["work"] / (dec["ms"] / 1e3) / 1e9 if dec["ms"] else 0.0
    st_gbs = st["work"] / (st["ms"] / 1e3) / 1e9 if st["ms"] else 0.0
    extend = {"qtok_s": n_ext * steps / (ext["ms"] / 1e3) if ext["ms"] else None,
              "tflops": ext_tflops, "frac_of_bf16_peak": ext_tflops / bf16_peak,
              "ms_per_step": ext["ms"] / steps, "launches_per_step": ext["launches"] / steps,
              "flop_per_step": ext["work"] / steps}
    decode = {"gbs": dec_gbs, "frac_of_hbm_peak": dec_gbs / hbm_peak,
              "ms_per_step": dec["ms"] / steps, "launches_per_step": dec["launches"] / steps,
              "bytes_per_step": dec["work"] / steps}
    if n_dec_launch_bytes is not None and dec["launches"] and n_dec_launch_bytes < L2_BYTES:
        decode["note"] = ("decode working set fits in L2; L2 is flushed between steps only, so "
                          "later decode steps of a step read KV that is partly L2-resident "
                          "(effective GB/s)")
    kv_store = {"gbs": st_gbs, "frac_of_hbm_peak": st_gbs / hbm_peak,
                "ms_per_step": st["ms"] / steps, "launches_per_step": st["launches"] / steps,
                "bytes_per_step": st["work"] / steps}
    return extend, decode, kv_store


def measure(wl, dev, steps, warmup, world, e2e=False, clocks=None):
    """Times `steps` runs of the whole workload (after `warmup` runs), inputs
    resident in HBM, L2 flushed between runs; optionally the end-to-end leg."""
    import torch
    import torch.distributed as dist

    from radix_tree_prefix_gb300 import rx, workloads
    from radix_tree_prefix_gb300.engine import (Engine, GatherInputs, OutputRing,
                                                PreparedInputs)

    layers = list(range(wl.num_layers))
    values = workloads.make_values(wl, dev, layers)
    source = GatherInputs(wl, values, layers)
    prepared = PreparedInputs(source)
    eng = Engine(wl, device=dev, inputs=prepared, layers=layers)
    trace = eng.run()                       # records the inputs of every batch/step
    prepared.freeze()
    torch.cuda.synchronize()
    rx.device_check()
    source.values = None                    # the stores are no longer needed
    del values
    n_ext = trace.prefilled
    n_dec = sum(len(w) for w in wl.waves) * wl.decode_steps
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    for _ in range(warmup):
        eng.run()
    torch.cuda.synchronize()
    if clocks is not None:
        time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    eng.timing = True
    eng.kernel_events = []
    launches0 = eng.gpu_launches
    step_ev = []
    stream = torch.cuda.current_stream()
    if clocks is not None:
        clocks.begin()
    wall0 = time.perf_counter()
    for _ in range(steps):
        flush.zero_()                                   # L2 flushed between steps
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        t = eng.run()
        e1.record(stream)
        step_ev.append((e0, e1))
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    if clocks is not None:
        clocks.end()
        clocks.result = clocks.stop()      # the sampler does not run during the e2e leg
    if world > 1:
        dist.barrier()
    assert t.as_tuple() == trace.as_tuple(), "timed steps made different cache decisions"
    rx.device_check()
    step_ms = [a.elapsed_time(b) for a, b in step_ev]
    ms = max_over_ranks(sum(step_ms) / len(step_ms), world, dev)
    out = {"wl": wl, "trace": trace, "n_ext": n_ext, "n_dec": n_dec, "ms": ms,
           "kinds": _kind_stats(eng.kernel_events, steps),
           "launches": eng.gpu_launches - launches0, "wall": wall, "e2e": None}
    eng.close()                             # its timing events are read
    if e2e:
        # host copies of every recorded input, then the device copies go
        host = PreparedInputs(source, host=True, ring=E2E_INPUT_RING)
        host.adopt(prepared)
        host.freeze()
        prepared.ext.clear()
        prepared.dec.clear()
        most = max([eng.max_extend_rows] + [len(w) * wl.decode_steps for w in wl.waves])
        del eng
        torch.cuda.empty_cache()
        hq, d = wl.num_q_heads, wl.head_dim
        # as many output buffers as fit in E2E_RING_BYTES (at least 4), so the
        # read-back of a batch's outputs can trail its kernels
        per = most * hq * (d + 1)
        ring = OutputRing(dev, per, slots=max(4, min(64, E2E_RING_BYTES // (4 * per))))
        eng2 = Engine(wl, device=dev, inputs=host, layers=layers, out_ring=ring)
        eng2.run()                                      # untimed first run
        torch.cuda.synchronize()
        host.h2d_bytes = 0
        ring.d2h_bytes = 0
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        # steps run back to back, as a serving loop runs them: the host makes
        # step n + 1's decisions while the GPU still works on step n; the
        # timed region ends once the last step's outputs are on the host
        host_s = []
        t0 = time.perf_counter()
        for _ in range(steps):
            flush.zero_()
            h0 = time.perf_counter()
            eng2.run()
            host_s.append(time.perf_counter() - h0)
        torch.cuda.synchronize()
        e2e_s = max_over_ranks((time.perf_counter() - t0) / steps, world, dev)
        rx.device_check()
        out["e2e"] = {"value": job_rate(n_ext + n_dec, e2e_s, world, dev), "unit": "query-tok/s",
                      "h2d_bytes_per_step": host.h2d_bytes // steps,
                      "d2h_bytes_per_step": ring.d2h_bytes // steps,
                      "ms_per_step": e2e_s * 1e3,
                      "host_ms_per_step": 1e3 * statistics.mean(host_s),
                      "copies": f"inputs from page-locked host memory up to {host.ring - 1} "
                                f"launch groups ahead on a side stream; every output (fp32 o and "
                                f"lse) read back through a ring of {ring.slots} device/host "
                                f"buffer pairs on another stream; steps back to back, one "
                                f"synchronize after the last"}
        eng2.close()
        del eng2
        ring.close()
        host.close()
    return out


def _summary(res, steps, hbm_peak, bf16_peak):
    wl = res["wl"]
    launch_bytes = None
    kinds = res["kinds"]
    if "decode" in kinds and kinds["decode"]["launches"]:
        per_launch = kinds["decode"]["work"] / kinds["decode"]["launches"]
        launch_bytes = per_launch / max(1, wl.decode_steps)
    extend, decode, kv_store = _rates(kinds, res["n_ext"], hbm_peak, bf16_peak, steps,
                                      launch_bytes)
    return extend, decode, kv_store


def only_kv_store(args, dev):
    """kv_store alone at the shape of the workload's largest extend batch:
    one layer's pool of the workload's slot count, the batch's new slots (from
    the host bookkeeping), seeded K/V rows; W untimed and K timed launches,
    L2 flushed before each."""
    import torch

    from radix_tree_prefix_gb300 import rx, workloads
    from radix_tree_prefix_gb300.engine import Engine

    wl = workloads.WORKLOADS[args.workload]()
    trace = Engine(wl).run()
    batch = max(trace.batches, key=lambda b: sum(len(r) - m for _, m, r in b))
    slots = np.concatenate([np.asarray(r[m:], dtype=np.int32) for _, m, r in batch])
    T, hkv, d = len(slots), wl.num_kv_heads, wl.head_dim
    g = torch.Generator(device=dev).manual_seed(1)
    kp = torch.zeros((1, hkv, wl.num_slots, d), dtype=torch.bfloat16, device=dev)
    vp = torch.zeros_like(kp)
    k = torch.randn((T, hkv, d), generator=g, device=dev).to(torch.bfloat16)
    v = torch.randn((T, hkv, d), generator=g, device=dev).to(torch.bfloat16)
    d_slots = torch.from_numpy(slots).to(dev)
    pool = rx.pool_desc(kp, vp)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    times = []
    for i in range(args.warmup + args.steps):
        flush.zero_()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        rx.kv_store(pool, 0, d_slots, k, v, stream)
        b.record(stream)
        times.append((a, b))
    torch.cuda.synchronize()
    rx.device_check()
    ms = statistics.mean(a.elapsed_time(b) for a, b in times[args.warmup:])
    nbytes = 4 * T * hkv * d * 2 + 4 * T
    hbm_peak, _, src = peaks()
    gbs = nbytes / (ms / 1e3) / 1e9
    print(json.dumps({"kernel": "kv_store_kernel", "workload": wl.name, "tokens": T,
                      "bytes_per_launch": nbytes, "ms_per_launch": ms, "gbs": gbs,
                      "frac_of_hbm_peak": gbs / hbm_peak, "peak_source": src,
                      "launches_timed": args.steps}), flush=True)


def main(argv=None):
    args = parse(argv)
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
    from radix_tree_prefix_gb300 import workloads

    if args.only == "kv_store":
        if rank == 0:
            only_kv_store(args, dev)
        return

    hbm_peak, bf16_peak, peak_src = peaks()
    # each replica takes its subtree-affine share (the whole workload on one GPU)
    full_wl = workloads.WORKLOADS[args.workload]()
    wl = workloads.shard(full_wl, rank, world)
    clocks = Clocks(local)          # started before warm-up: its start-up is not timed
    res = measure(wl, dev, args.steps, args.warmup, world, e2e=not args.no_e2e, clocks=clocks)
    clk = clocks.result
    torch.cuda.empty_cache()
    n_ext, n_dec = res["n_ext"], res["n_dec"]
    q_per_step = n_ext + n_dec
    value = job_rate(q_per_step, res["ms"] / 1000.0, world, dev)
    extend, decode, kv_store = _summary(res, args.steps, hbm_peak, bf16_peak)
    if extend["ms_per_step"] >= decode["ms_per_step"]:
        roof = {"kernel": "rx_extend_attention", "bound": "tensor", "achieved": extend["tflops"],
                "peak": bf16_peak, "unit": "TFLOP/s", "frac": extend["frac_of_bf16_peak"],
                "traffic": TRAFFIC.get((wl.name, "rx_extend_attention")),
                "peak_source": f"{peak_src} bf16_tflops (burst)"}
    else:
        roof = {"kernel": "rx_decode_attention", "bound": "hbm", "achieved": decode["gbs"],
                "peak": hbm_peak, "unit": "GB/s", "frac": decode["frac_of_hbm_peak"],
                "traffic": TRAFFIC.get((wl.name, "rx_decode_attention")),
                "peak_source": f"{peak_src} hbm_gbs"}

    configs = {}
    if not args.no_configs and world == 1:
        for name in SIDE_WORKLOADS:
            if name == wl.name:
                continue
            side = measure(workloads.WORKLOADS[name](), dev, SIDE_STEPS, 3, 1)
            e, dcd, st = _summary(side, SIDE_STEPS, hbm_peak, bf16_peak)
            configs[name] = {"ms_per_step": side["ms"],
                             "query_tokens_per_step": side["n_ext"] + side["n_dec"],
                             "value": (side["n_ext"] + side["n_dec"]) / (side["ms"] / 1e3),
                             "steps": SIDE_STEPS, "warmup": 3,
                             "extend": e, "decode": dcd, "kv_store": st}
            del side
            torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and not args.no_cpu and world == 1:
        cpu = oracle_rate(wl)
        cpu.pop("seconds", None)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "query-tok/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["ms"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": config_of(full_wl, world),
            "detail": {"query_tokens_per_step": q_per_step, "extend_query_tokens": n_ext,
                       "decode_query_tokens": n_dec,
                       "wall_s_timed_region_incl_flush": res["wall"]},
            "extend": extend, "decode": decode, "kv_store": kv_store, "roofline": roof,
            "cpu_baseline": cpu, "e2e": res["e2e"], "gpu_launches": res["launches"],
            "clocks": clk, "configs": configs,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

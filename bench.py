"""Benchmark of paged GDN prefill and decode on one GB300 (or N replicas).

One step = the long-context prefill workload: gdn_paged_prefill_slots plus the
chunked paged prefill of 4 sequences x 65,536 new tokens (H = 32, K = V = 128,
page_size 1152, state stored at all 57 page ends of every sequence).  The
decode batch (B = 256, H = 32, page_size 1024, 10,000-page pool) is timed the
same way as a second measurement: gdn_paged_decode_slots + one decode step.

Timing: W untimed warm-up steps, then exactly K steps between a barrier and a
device synchronize on both sides, CUDA events on the launching stream, max
over ranks.  Every input is larger than L2 (prefill streams 8.6 GB of
q/k/v/o, decode 1.08 GB of state), so no L2 flush is needed.  N > 1 runs N
independent replicas (one per GPU, no collective on the data path).

--impl reference times the fp64 CPU oracle (the only reference this method
has) on the host cores over a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "GDN paged prefill tok/s + decode seq/s on 1 GB300; % HBM / tensor roofline"
UNIT = "tok/s"
SCALE = 128 ** -0.5
K = V = 128
FLOP_PER_TOKEN_HEAD = 10 * 64 * 128 + 6 * 128 * 128      # 180,224 (tensor-core contractions)
BYTES_PER_TOKEN_HEAD = 2 * (2 * K + 2 * V) + 8           # q, k, v, o bf16 + g, beta fp32 = 1032
STATE_BYTES = V * K * 4                                   # one (row, head) state, fp32
DECODE_BYTES_PER_SEQ_HEAD = 2 * STATE_BYTES + 2 * (2 * K + 2 * V) + 8   # 132,104
DECODE_BF16_BYTES_PER_SEQ_HEAD = 2 * (V * K * 2) + 2 * (2 * K + 2 * V) + 8   # 66,568: bf16 state pool

# DRAM bytes (read + write) of one paged prefill call per new token, over all heads:
# ncu capture of the 4 x 8192-token case (ut_kernel 0.621 GB + prefill_kernel 1.516 GB
# for 32,768 tokens); the traffic grows in proportion to the tokens.
PREFILL_TRAFFIC_PER_TOKEN = 2.137e9 / 32768
TRAFFIC_SOURCE = "ncu dram__bytes_read+write of 4x8192-token call, scaled by tokens"
PREFILL = dict(S=4, L=65536, H=32, page_size=1152, num_pages=256)
DECODE = dict(B=256, H=32, page_size=1024, num_pages=10000)
NOMINAL_HBM_GBS = 8000.0  # GB300 HBM3e, nominal (the roofline's peak is the measured copy rate)


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def prefill_config(tokens_per_seq, world):
    """The `config` of the prefill line, the same for both arms."""
    full = tokens_per_seq == PREFILL["L"]
    return {"workload": "long-context paged prefill: 4 seqs x %d new tokens, H=32, K=V=128, page_size=1152, "
                        "state stored at every page end (step = slots + prefill)%s"
                        % (tokens_per_seq, "" if full else " [reduced size: not a headline run]"),
            "tokens_per_step": PREFILL["S"] * tokens_per_seq,
            "l2": "inputs larger than L2 (streamed q/k/v/o per step), no flush",
            "parallelism": "replicas" if world > 1 else "single GPU"}


class Replicas:
    """Timing coordination of N independent replicas, one process per GPU
    (no collective on the data path): a barrier on both sides of every timed
    region and the maximum of a per-rank time over the ranks.  ``dist`` is
    torch.distributed with an initialised process group, or None for one
    process; ``device`` is where the reduction tensor lives (the GPU with NCCL,
    "cpu" with gloo)."""

    def __init__(self, dist=None, device="cpu"):
        self.dist = dist
        self.device = device

    def barrier(self):
        if self.dist is not None:
            self.dist.barrier()

    def max(self, x):
        if self.dist is None:
            return x
        t = torch.tensor([x], dtype=torch.float64, device=self.device)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())


def launch_env():
    """(rank, world size, local rank) from the launcher's environment; one
    process when absent."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def run_gpu(args, rank, world, local_rank):
    import gated_deltanet_paged_gb300 as gdn
    from gated_deltanet_paged_gb300 import workloads

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    replicas = Replicas(dist, dev)
    barrier, max_over_ranks = replicas.barrier, replicas.max

    hbm, bf16, peak_kind = peaks()
    stream = torch.cuda.current_stream(dev)

    # ---- prefill workload (one replica per rank) ----
    line = {}
    launches = 0
    if args.workload in ("all", "prefill"):
        launches += _bench_prefill(args, gdn, workloads, dev, stream, barrier, max_over_ranks, rank, world,
                                   hbm, bf16, peak_kind, line)
    if args.workload in ("all", "decode"):
        launches += _bench_decode(args, gdn, workloads, dev, stream, barrier, max_over_ranks, rank, world, hbm,
                                  line)
    if args.workload in ("all", "layers"):
        launches += _bench_layers(args, gdn, workloads, dev, stream, barrier, max_over_ranks, world, hbm, line)
    if args.workload in ("all", "configs"):
        launches += _bench_configs(args, gdn, workloads, dev, stream, hbm, bf16, line)
    line["gpu_launches"] = launches
    if rank == 0 and not args.no_cpu_baseline and args.workload in ("all", "prefill"):
        line["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    line["summary"] = summary(line)
    if dist is not None:
        dist.destroy_process_group()
    return line


def _bench_prefill(args, gdn, workloads, dev, stream, barrier, max_over_ranks, rank, world, hbm, bf16, peak_kind,
                   line):
    wp = workloads.long_context(dev, L=args.prefill_tokens, decode_steps=128, seed=1238 + rank)
    pre = wp.calls[0]
    pool = wp.pool
    T, H = pre.q.shape[0], pre.q.shape[1]
    o = torch.empty(T, H, V, dtype=torch.bfloat16, device=dev)
    stores = sum(-(-(int(l)) // PREFILL["page_size"]) for l in wp.seq_lens.tolist())  # page ends + final
    prefill_bytes = T * H * BYTES_PER_TOKEN_HEAD + stores * H * STATE_BYTES
    prefill_flops = T * H * FLOP_PER_TOKEN_HEAD
    slot_out = gdn.gdn_paged_prefill_slots(pre.cu_seqlens, pre.page_indptr, pre.page_indices, pre.last_page_len,
                                           pre.page_size)
    # Workspace of the chunk-local phase (one 64 x 64 fp16 tile per chunk and
    # head), allocated once outside the timed region like any caller would.
    ws = torch.empty(gdn.gdn_prefill_workspace_bytes(pre.cu_seqlens.numel() - 1, T, H), dtype=torch.uint8,
                     device=dev)

    def prefill_step(ev=None):
        gdn.gdn_paged_prefill_slots(pre.cu_seqlens, pre.page_indptr, pre.page_indices, pre.last_page_len,
                                    pre.page_size, out=slot_out)
        if ev is not None:
            ev[0].record(stream)
        gdn.gdn_chunk_gated_delta_rule_paged(pre.q, pre.k, pre.v, pre.g, pre.beta, pre.cu_seqlens, pool,
                                             pre.page_indices, pre.page_indptr, pre.page_size, pre.last_page_len,
                                             scale=SCALE, slots=slot_out, o=o, workspace=ws)
        if ev is not None:
            ev[1].record(stream)

    for _ in range(args.warmup):
        prefill_step()
    torch.cuda.synchronize(dev)
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        barrier()
        torch.cuda.synchronize(dev)
        start.record(stream)
        for i in range(args.steps):
            prefill_step(kev[i])
        stop.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
    ms_prefill = max_over_ranks(start.elapsed_time(stop) / args.steps)
    kernel_ms = statistics.mean(a.elapsed_time(b) for a, b in kev)
    clocks = clk.summary()
    launches = 4 * args.steps  # slots, slot map, chunk-local kernel, state chain

    # ---- e2e: host buffers, copies inside the timed region ----
    # Every step copies its own inputs from pinned host memory and reads its
    # output back, as a serving loop would: the steps are pipelined over three
    # kinds of streams (input copies split over three copy streams, the call on
    # the main stream, the read-back on its own), with the device-side inputs
    # and outputs double-buffered, so step i+1's inputs travel while step i
    # computes and step i-1's output comes back.
    e2e = None
    if not args.no_e2e:
        names = ("q", "k", "v", "g", "beta")
        # one pinned copy of the inputs (read-only on the host) and one output
        # buffer (the read-backs run in order on one stream)
        host = {n: getattr(pre, n).cpu().pin_memory() for n in names}
        host_o = torch.empty(T, H, V, dtype=torch.bfloat16).pin_memory()
        dbuf = [{n: torch.empty_like(getattr(pre, n)) for n in names} for _ in range(2)]
        dev_o = [torch.empty(T, H, V, dtype=torch.bfloat16, device=dev) for _ in range(2)]
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = host_o.numel() * host_o.element_size()
        s_in = [torch.cuda.Stream(dev) for _ in range(3)]
        s_out = torch.cuda.Stream(dev)

        def e2e_run(nsteps, marks=None):
            """nsteps pipelined steps; marks (optional) collects per-step events."""
            ev = lambda: torch.cuda.Event(enable_timing=marks is not None)
            done_call, done_out = [None] * nsteps, [None] * nsteps
            for i in range(nsteps):
                b = i & 1
                ins = []
                for j, n in enumerate(("q", "k", "v")):  # the large tensors, one copy stream each
                    st = s_in[j]
                    with torch.cuda.stream(st):
                        if i >= 2:
                            st.wait_event(done_call[i - 2])  # buffer b free: call i-2 has read it
                        if marks is not None and j == 0:
                            e0 = ev(); e0.record(st)
                        dbuf[b][n].copy_(host[n], non_blocking=True)
                        if n == "v":
                            dbuf[b]["g"].copy_(host["g"], non_blocking=True)
                            dbuf[b]["beta"].copy_(host["beta"], non_blocking=True)
                        e = ev(); e.record(st); ins.append(e)
                for e in ins:
                    stream.wait_event(e)
                if i >= 2:
                    stream.wait_event(done_out[i - 2])  # output buffer b read back
                if marks is not None:
                    c0 = ev(); c0.record(stream)
                gdn.gdn_chunk_gated_delta_rule_paged(
                    dbuf[b]["q"], dbuf[b]["k"], dbuf[b]["v"], dbuf[b]["g"], dbuf[b]["beta"], pre.cu_seqlens, pool,
                    pre.page_indices, pre.page_indptr, pre.page_size, pre.last_page_len, scale=SCALE, o=dev_o[b],
                    workspace=ws)
                done_call[i] = ev(); done_call[i].record(stream)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(done_call[i])
                    host_o.copy_(dev_o[b], non_blocking=True)
                    done_out[i] = ev(); done_out[i].record(s_out)
                if marks is not None:
                    marks.append((e0, ins, c0, done_call[i], done_out[i]))
            for st in s_in + [s_out]:
                stream.wait_stream(st)

        e2e_run(max(3, args.warmup))  # first touches of the pinned buffers are slow
        torch.cuda.synchronize(dev)
        e2e_steps = max(2, min(args.steps, 6))
        barrier()
        torch.cuda.synchronize(dev)
        marks = []
        start.record(stream)
        for st in s_in + [s_out]:
            st.wait_stream(stream)
        e2e_run(e2e_steps, marks)
        stop.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
        ms_e2e = max_over_ranks(start.elapsed_time(stop) / e2e_steps)
        mean = lambda xs: statistics.mean(xs)
        e2e = {"value": T * world / (ms_e2e * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e,
               "pipelined": "device inputs and outputs double-buffered; input copies on 3 streams, read-back on its own",
               "parts_ms": {"h2d": mean(max(m[0].elapsed_time(e) for e in m[1]) for m in marks),
                            "call": mean(m[2].elapsed_time(m[3]) for m in marks),
                            "d2h": mean(m[3].elapsed_time(m[4]) for m in marks)}}
        launches += 3 * e2e_steps  # timed steps: slot map, chunk-local kernel, state chain
        del host, host_o, dbuf, dev_o

    value = T * world / (ms_prefill * 1e-3)
    achieved = prefill_bytes / (kernel_ms * 1e-3) / 1e9
    line.update({
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_prefill,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "precision": "bf16 q/k/v/o, fp32 g/beta/state, fp16 tensor-core operands with fp32 accumulation",
        "data": "synthetic (seeded; q,k L2-normalised bf16, v bf16, g=-softplus(N), beta=sigmoid(N))",
        "config": prefill_config(args.prefill_tokens, world),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "frac_of_nominal_8000": achieved / NOMINAL_HBM_GBS,
                     "traffic": PREFILL_TRAFFIC_PER_TOKEN * T, "traffic_source": TRAFFIC_SOURCE,
                     "kernel": "paged prefill call (slot map + chunk-local kernel + state chain)",
                     "kernel_ms": kernel_ms,
                     "algorithmic_bytes": prefill_bytes, "peak_kind": peak_kind},
        "tensor": {"achieved_tflops": prefill_flops / (kernel_ms * 1e-3) / 1e12, "peak_tflops": bf16,
                   "frac": prefill_flops / (kernel_ms * 1e-3) / 1e12 / bf16, "flops_per_launch": prefill_flops},
        "clocks": clocks,
    })
    if e2e is not None:
        line["e2e"] = e2e
    del o

    # ---- the workload's decode phase: 128 steps at B = 4 on the prefilled pool ----
    decs = wp.calls[1:]
    dslots = gdn.gdn_paged_decode_slots(decs[0].page_indptr, decs[0].page_indices, decs[0].last_page_len)
    od = torch.empty(PREFILL["S"], H, V, dtype=torch.bfloat16, device=dev)

    def decode_phase():
        for c in decs:
            gdn.gdn_paged_decode_slots(c.page_indptr, c.page_indices, c.last_page_len, out=dslots)
            gdn.gdn_gated_delta_rule_decode_paged(c.q, c.k, c.v, c.g, c.beta, pool, c.page_indices, c.page_indptr,
                                                  c.last_page_len, scale=SCALE, slots=dslots, o=od)

    decode_phase()  # warm-up (in place: repeats rewrite the same rows)
    reps = 5

    def time_phase(run):
        pev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        torch.cuda.synchronize(dev)
        for a_, b_ in pev:
            a_.record(stream)
            run()
            b_.record(stream)
        torch.cuda.synchronize(dev)
        return statistics.median(a_.elapsed_time(b_) for a_, b_ in pev)

    eager_ms = time_phase(decode_phase)
    # the same 128 steps captured once as a CUDA graph and replayed: the device
    # time of a step without the host's per-call cost
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        decode_phase()
    stream.wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        decode_phase()
    graph.replay()
    graph_ms = time_phase(graph.replay)
    del graph

    # the same steps with the decode call deriving its rows from the page table
    # (no slots argument): one launch per step
    def decode_phase_fused():
        for c in decs:
            gdn.gdn_gated_delta_rule_decode_paged(c.q, c.k, c.v, c.g, c.beta, pool, c.page_indices, c.page_indptr,
                                                  c.last_page_len, scale=SCALE, o=od)

    with torch.cuda.stream(side):
        decode_phase_fused()
    stream.wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        decode_phase_fused()
    graph.replay()
    fused_ms = time_phase(graph.replay)
    del graph
    step_bytes = PREFILL["S"] * H * DECODE_BYTES_PER_SEQ_HEAD
    us_step = 1e3 * graph_ms / len(decs)
    line["long_context_decode"] = {
        "workload": "the long-context workload's decode phase: 128 decode steps at B=4, H=32, on the prefilled "
                    "pool (step = decode slots + decode; last_page_len 1025..1152, in place), replayed as one "
                    "captured CUDA graph",
        "us_per_step": us_step, "eager_us_per_step": 1e3 * eager_ms / len(decs),
        "rows_from_page_table_us_per_step": 1e3 * fused_ms / len(decs),
        "value": PREFILL["S"] / (us_step * 1e-6), "unit": "seq/s",
        "roofline": {"bound": "latency", "achieved": step_bytes / (us_step * 1e-6) / 1e9, "peak": hbm,
                     "unit": "GB/s", "frac": step_bytes / (us_step * 1e-6) / 1e9 / hbm,
                     "algorithmic_bytes_per_step": step_bytes},
        "reps": reps}
    launches += 2 * len(decs) * 2 * reps + len(decs) * reps  # eager and graph phases, one-launch graph
    return launches


def _event_median_ms(stream, fn, reps):
    """Median CUDA-event time of fn() on the stream over reps calls (each call
    bracketed by its own pair of events)."""
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    torch.cuda.synchronize()
    for a_, b_ in ev:
        a_.record(stream)
        fn()
        b_.record(stream)
    torch.cuda.synchronize()
    return statistics.median(a_.elapsed_time(b_) for a_, b_ in ev)


def _checkpoint_layout(prefix, lens, N):
    """Checkpoints per sequence, (prefix + len) // N - prefix // N ("Slot
    arguments of chunk_gated_delta_rule"), laid out densely: (cu_starts, total)."""
    counts = (prefix + lens) // N - prefix // N
    starts = np.concatenate([[0], np.cumsum(counts)[:-1]]).astype(np.int32)
    return starts, int(counts.sum())


def _bench_configs(args, gdn, workloads, dev, stream, hbm, bf16, line):
    """The other workloads of the method's pages: the tiny two-sequence case
    and the worked 2500-token example (latency of one call), and the mixed
    chunked-prefill batch through the general slot API (tok/s with both
    roofline fractions, computed from its seeded draw)."""
    out = {}
    launches = 0
    todev = lambda t: t.to(dev)
    reps = 50

    # tiny: the prefix call untimed, then the main prefill call and the decode step
    w = workloads.tiny("cpu")
    pool = todev(w.pool)
    c0, c1, cd = w.calls
    ws = torch.empty(gdn.gdn_prefill_workspace_bytes(2, 137, w.H), dtype=torch.uint8, device=dev)

    def pf(c):
        return lambda: gdn.gdn_chunk_gated_delta_rule_paged(
            todev_c[c].q, todev_c[c].k, todev_c[c].v, todev_c[c].g, todev_c[c].beta, todev_c[c].cu_seqlens, pool,
            todev_c[c].page_indices, todev_c[c].page_indptr, todev_c[c].page_size, todev_c[c].last_page_len,
            scale=SCALE, workspace=ws, o=outs[c])

    class _C:
        pass

    def move(c):
        m = _C()
        for n in ("q", "k", "v", "g", "beta", "page_indptr", "page_indices", "last_page_len"):
            setattr(m, n, todev(getattr(c, n)))
        if hasattr(c, "cu_seqlens"):
            m.cu_seqlens = todev(c.cu_seqlens)
        m.page_size = c.page_size
        return m

    todev_c = {i: move(c) for i, c in enumerate(w.calls)}
    outs = {0: torch.empty(64, w.H, V, dtype=torch.bfloat16, device=dev),
            1: torch.empty(137, w.H, V, dtype=torch.bfloat16, device=dev)}
    pf(0)()
    ms_pre = _event_median_ms(stream, pf(1), reps)
    dc = todev_c[2]
    od = torch.empty(2, w.H, V, dtype=torch.bfloat16, device=dev)
    ms_dec = _event_median_ms(stream, lambda: gdn.gdn_gated_delta_rule_decode_paged(
        dc.q, dc.k, dc.v, dc.g, dc.beta, pool, dc.page_indices, dc.page_indptr, dc.last_page_len, scale=SCALE,
        o=od), reps)
    out["tiny"] = {"workload": w.name, "prefill_call_us": 1e3 * ms_pre, "decode_call_us": 1e3 * ms_dec,
                   "unit": "us per call (median of %d, CUDA events)" % reps}
    launches += reps * 4  # prefill: slot map, chunk-local, chain; decode: one kernel

    # worked example: the 2048-token prefix call untimed, then the 452-token call
    w = workloads.worked_example("cpu")
    pool = todev(w.pool)
    todev_c = {i: move(c) for i, c in enumerate(w.calls)}
    outs = {0: torch.empty(2048, w.H, V, dtype=torch.bfloat16, device=dev),
            1: torch.empty(452, w.H, V, dtype=torch.bfloat16, device=dev)}
    ws = torch.empty(gdn.gdn_prefill_workspace_bytes(1, 2048, w.H), dtype=torch.uint8, device=dev)
    pf(0)()
    ms_w = _event_median_ms(stream, pf(1), reps)
    out["worked_example"] = {"workload": w.name, "prefill_call_us": 1e3 * ms_w,
                             "value": 452 / (ms_w * 1e-3), "unit": "tok/s (452 new tokens per call)"}
    launches += reps * 3

    # mixed chunked prefill through the general slot API, checkpoints into a separate buffer
    w = workloads.mixed_prefill("cpu")
    c = move(w.calls[0])
    P, L = w.prefix_lens.numpy(), w.seq_lens.numpy()
    N = w.checkpoint_every
    ccs, total = _checkpoint_layout(P, L, N)
    pool = todev(w.pool)
    ck = torch.zeros(total, w.H, V, K, dtype=torch.float32, device=dev)
    cki = torch.arange(total, dtype=torch.int32, device=dev)
    ccs_d = torch.as_tensor(ccs, device=dev)
    T, H = c.q.shape[0], w.H
    S = len(L)
    ws = torch.empty(gdn.gdn_prefill_workspace_bytes(S, T, H), dtype=torch.uint8, device=dev)
    om = torch.empty(T, H, V, dtype=torch.bfloat16, device=dev)
    slots = gdn.gdn_paged_prefill_slots(c.cu_seqlens, c.page_indptr, c.page_indices, c.last_page_len, w.page_size)

    def mixed_step(ev=None):
        gdn.gdn_paged_prefill_slots(c.cu_seqlens, c.page_indptr, c.page_indices, c.last_page_len, w.page_size,
                                    out=slots)
        gdn.gdn_chunk_gated_delta_rule(
            c.q, c.k, c.v, c.g, c.beta, c.cu_seqlens, scale=SCALE, initial_state=pool,
            state_indices=slots["state_indices"], output_state=pool,
            output_state_indices=slots["output_state_indices"], state_checkpoints=ck,
            checkpoint_state_indices=cki, checkpoint_cu_starts=ccs_d, prefix_lens=slots["prefix_lens"],
            checkpoint_every_n_tokens=N, o=om, workspace=ws)

    for _ in range(3):
        mixed_step()
    with ClockSampler(dev.index) as clk:
        ms_m = _event_median_ms(stream, mixed_step, 20)
    reads = int(((P > 0) & (L > 0)).sum())
    writes = int((L > 0).sum()) + total
    mbytes = int(L.sum()) * H * BYTES_PER_TOKEN_HEAD + (reads + writes) * H * STATE_BYTES
    mflops = int(L.sum()) * H * FLOP_PER_TOKEN_HEAD
    ach = mbytes / (ms_m * 1e-3) / 1e9
    tf = mflops / (ms_m * 1e-3) / 1e12
    out["mixed_prefill"] = {
        "workload": w.name + " (general slot API, checkpoints every 896 tokens into a separate buffer; "
                             "step = slots + prefill)",
        "new_tokens": int(L.sum()), "longest": int(L.max()), "state_reads": reads, "state_writes": writes,
        "ms_per_step": ms_m, "value": int(L.sum()) / (ms_m * 1e-3), "unit": "tok/s",
        "roofline": {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
                     "algorithmic_bytes": mbytes},
        "tensor": {"achieved_tflops": tf, "peak_tflops": bf16, "frac": tf / bf16, "flops_per_step": mflops},
        "clocks": clk.summary()}
    launches += 20 * 4
    line["configs"] = out
    return launches


def _bench_decode(args, gdn, workloads, dev, stream, barrier, max_over_ranks, rank, world, hbm, line):
    H = DECODE["H"]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wd = workloads.decode_batch(dev, seed=1236 + rank, max_ctx=args.decode_max_ctx, num_pages=args.decode_pages)
    dc = wd.calls[0]
    dpool = wd.pool
    od = torch.empty(DECODE["B"], H, V, dtype=torch.bfloat16, device=dev)
    dslots = gdn.gdn_paged_decode_slots(dc.page_indptr, dc.page_indices, dc.last_page_len)

    def decode_step(pool, ev=None):
        gdn.gdn_paged_decode_slots(dc.page_indptr, dc.page_indices, dc.last_page_len, out=dslots)
        if ev is not None:
            ev[0].record(stream)
        gdn.gdn_gated_delta_rule_decode_paged(dc.q, dc.k, dc.v, dc.g, dc.beta, pool, dc.page_indices,
                                              dc.page_indptr, dc.last_page_len, scale=SCALE, slots=dslots, o=od)
        if ev is not None:
            ev[1].record(stream)

    dsteps = max(args.steps, 200)

    def timed(pool):
        for _ in range(max(args.warmup, 3)):
            decode_step(pool)
        dev_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(dsteps)]
        with ClockSampler(dev.index) as clk:
            barrier()
            torch.cuda.synchronize(dev)
            start.record(stream)
            for i in range(dsteps):
                decode_step(pool, dev_ev[i])
            stop.record(stream)
            torch.cuda.synchronize(dev)
            barrier()
        return (max_over_ranks(start.elapsed_time(stop) / dsteps),
                statistics.mean(a.elapsed_time(b) for a, b in dev_ev), clk.summary())

    ms_decode, dkernel_ms, dclocks = timed(dpool)

    # Copy-on-write forks of 256 pool rows (2 MB each) into rows no sequence
    # uses: the row utility's bit-exact copy, HBM-bound.
    used = set(dslots["initial_state_indices"].tolist()) | set(dslots["output_state_indices"].tolist())
    free = [r for r in torch.randperm(dpool.shape[0], generator=torch.Generator().manual_seed(1240)).tolist()
            if r not in used][:DECODE["B"]]
    csrc = dslots["output_state_indices"].clone()
    cdst = torch.tensor(free, dtype=torch.int32, device=dev)
    for _ in range(3):
        gdn.gdn_pool_copy_rows(dpool, csrc, cdst)
    cev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(50)]
    torch.cuda.synchronize(dev)
    for a_, b_ in cev:
        a_.record(stream)
        gdn.gdn_pool_copy_rows(dpool, csrc, cdst)
        b_.record(stream)
    torch.cuda.synchronize(dev)
    copy_ms = statistics.mean(a_.elapsed_time(b_) for a_, b_ in cev)
    copy_bytes = 2 * DECODE["B"] * H * STATE_BYTES
    copy_ach = copy_bytes / (copy_ms * 1e-3) / 1e9
    decode_bytes = DECODE["B"] * H * DECODE_BYTES_PER_SEQ_HEAD
    ach = decode_bytes / (dkernel_ms * 1e-3) / 1e9
    dec = {"metric": "decode seq/s", "value": DECODE["B"] * world / (ms_decode * 1e-3), "unit": "seq/s",
           "ms_per_step": ms_decode, "kernel_ms": dkernel_ms, "steps": dsteps,
           "workload": "paged decode batch: B=256, H=32, page_size=1024, ctx U{2..32768}, "
                       "25% open a page, 10,000-page pool (step = decode slots + decode)",
           "roofline": {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
                        "frac_of_nominal_8000": ach / NOMINAL_HBM_GBS,
                        "algorithmic_bytes": decode_bytes},
           "clocks": dclocks,
           "pool_copy_rows": {"rows": DECODE["B"], "bytes_per_call": copy_bytes, "kernel_ms": copy_ms,
                              "roofline": {"bound": "hbm", "achieved": copy_ach, "peak": hbm, "unit": "GB/s",
                                           "frac": copy_ach / hbm}}}
    # The same batch on a bf16 state pool (the fp32 pool's values cut to bf16):
    # half the state bytes, fp32 arithmetic on the chip.
    bpool = (dpool.view(torch.int32) >> 16).to(torch.int16).view(torch.bfloat16)
    ms_b, kms_b, clk_b = timed(bpool)
    del bpool
    bytes_b = DECODE["B"] * H * DECODE_BF16_BYTES_PER_SEQ_HEAD
    ach_b = bytes_b / (kms_b * 1e-3) / 1e9
    dec["bf16_state_pool"] = {
        "value": DECODE["B"] * world / (ms_b * 1e-3), "unit": "seq/s", "ms_per_step": ms_b, "kernel_ms": kms_b,
        "steps": dsteps, "roofline": {"bound": "hbm", "achieved": ach_b, "peak": hbm, "unit": "GB/s",
                                      "frac": ach_b / hbm, "algorithmic_bytes": bytes_b},
        "clocks": clk_b}
    if "metric" in line:
        line["decode"] = dec
    else:  # decode-only run: the decode measurement is the line
        line.update({"metric": METRIC, "value": dec["value"], "unit": "seq/s", "n_gpus": world, "steps": dsteps,
                     "warmup": max(args.warmup, 3), "ms_per_step": ms_decode, "higher_is_better": True,
                     "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded)",
                     "config": {"workload": dec["workload"]}, "roofline": dec["roofline"], "clocks": dec["clocks"],
                     "bf16_state_pool": dec["bf16_state_pool"], "pool_copy_rows": dec["pool_copy_rows"]})
    return 4 * dsteps  # slots + decode, fp32 and bf16 pools (the row-copy timing is a side measurement)


def _bench_layers(args, gdn, workloads, dev, stream, barrier, max_over_ranks, world, hbm, line):
    """Multi-layer model steps: one slots call per step shared by L = 32
    layers, each layer with its own state pool and inputs, run eagerly (one
    binding call per layer) and as one captured CUDA graph replayed per step.
    Between two steps every layer's rows pass once, 1 GB or more, so L2 holds
    nothing of a layer from one step to the next (no flush)."""
    L = 32
    steps = max(args.steps, 10)
    res = {}
    launches = 0
    for name, make in (("decode_B256", lambda: workloads.decode_layers(dev, L=L, B=256, seed=1241 + 10 * world)),
                       ("decode_B8", lambda: workloads.decode_layers(dev, L=L, B=8, seed=1243 + 10 * world)),
                       ("prefill_4x8192", lambda: workloads.prefill_layers(dev, L=L, seed=1244 + 10 * world))):
        st = make()
        c0 = st.calls[0]
        H = st.H
        if isinstance(c0, workloads.DecodeCall):
            B = c0.q.shape[0]
            slots = gdn.gdn_paged_decode_slots(c0.page_indptr, c0.page_indices, c0.last_page_len)
            outs = [torch.empty(B, H, V, dtype=torch.bfloat16, device=dev) for _ in range(L)]

            def step():
                gdn.gdn_paged_decode_slots(c0.page_indptr, c0.page_indices, c0.last_page_len, out=slots)
                for l, c in enumerate(st.calls):
                    gdn.gdn_gated_delta_rule_decode_paged(c.q, c.k, c.v, c.g, c.beta, st.pools[l], c.page_indices,
                                                          c.page_indptr, c.last_page_len, scale=SCALE, slots=slots,
                                                          o=outs[l])
            units, unit = B, "seq"
            layer_bytes = B * H * DECODE_BYTES_PER_SEQ_HEAD
        else:
            T = c0.q.shape[0]
            S = c0.cu_seqlens.numel() - 1
            slots = gdn.gdn_paged_prefill_slots(c0.cu_seqlens, c0.page_indptr, c0.page_indices, c0.last_page_len,
                                                c0.page_size)
            outs = [torch.empty(T, H, V, dtype=torch.bfloat16, device=dev) for _ in range(L)]
            ws = torch.empty(gdn.gdn_prefill_workspace_bytes(S, T, H), dtype=torch.uint8, device=dev)

            def step():
                gdn.gdn_paged_prefill_slots(c0.cu_seqlens, c0.page_indptr, c0.page_indices, c0.last_page_len,
                                            c0.page_size, out=slots)
                for l, c in enumerate(st.calls):
                    gdn.gdn_chunk_gated_delta_rule_paged(c.q, c.k, c.v, c.g, c.beta, c.cu_seqlens, st.pools[l],
                                                         c.page_indices, c.page_indptr, c.page_size,
                                                         c.last_page_len, scale=SCALE, slots=slots, o=outs[l],
                                                         workspace=ws)
            units, unit = T, "tok"
            stores = S * -(-(T // S) // c0.page_size)
            layer_bytes = T * H * BYTES_PER_TOKEN_HEAD + stores * H * STATE_BYTES
        per_step = (1 + L) if unit == "seq" else (1 + 3 * L)  # slots + per layer decode / (slot map, ut, chain)

        def timed(run):
            for _ in range(max(args.warmup, 3)):
                run()
            start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with ClockSampler(dev.index) as clk:
                barrier()
                torch.cuda.synchronize(dev)
                start.record(stream)
                for _ in range(steps):
                    run()
                stop.record(stream)
                torch.cuda.synchronize(dev)
                barrier()
            return max_over_ranks(start.elapsed_time(stop) / steps), clk.summary()

        eager_ms, clk_e = timed(step)
        # capture one step (slots + all layers) after an eager warm-up on the capture side stream
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step()
        stream.wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        graph_ms, clk_g = timed(graph.replay)
        ach = L * layer_bytes / (graph_ms * 1e-3) / 1e9
        res[name] = {"workload": st.name, "layers": L, "steps": steps,
                     "eager_ms_per_step": eager_ms, "graph_ms_per_step": graph_ms,
                     "graph_us_per_layer": 1e3 * graph_ms / L,
                     "value": units * world / (graph_ms * 1e-3), "unit": "%s/s through all %d layers" % (unit, L),
                     "roofline": {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
                        "frac_of_nominal_8000": ach / NOMINAL_HBM_GBS,
                                  "algorithmic_bytes_per_step": L * layer_bytes},
                     "launches_per_step": per_step, "clocks": {"eager": clk_e, "graph": clk_g}}
        launches += 2 * steps * per_step
        del graph, st, outs, slots, step
        torch.cuda.synchronize(dev)
        torch.cuda.empty_cache()
    line["layer_step"] = res
    if "metric" not in line:  # layers-only run: the 256-sequence decode step is the line
        d = res["decode_B256"]
        line.update({"metric": METRIC, "value": d["value"], "unit": "seq/s", "n_gpus": world, "steps": steps,
                     "warmup": max(args.warmup, 3), "ms_per_step": d["graph_ms_per_step"], "higher_is_better": True,
                     "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded)",
                     "config": {"workload": d["workload"]}, "roofline": d["roofline"], "clocks": d["clocks"]["graph"]})
    return launches


def summary(line):
    """The headline figures of every measured workload in one short object,
    printed last so that a reader of the line's tail sees them all."""
    def get(d, *path):
        for p_ in path:
            if not isinstance(d, dict) or p_ not in d:
                return None
            d = d[p_]
        return round(d, 4) if isinstance(d, float) else d

    return {
        "prefill_long_context_tok_s": get(line, "value") if "tensor" in line else None,
        "prefill_ms": get(line, "roofline", "kernel_ms"),
        "prefill_tensor_frac": get(line, "tensor", "frac"),
        "prefill_hbm_frac": get(line, "roofline", "frac") if "tensor" in line else None,
        "decode_seq_s": get(line, "decode", "value"),
        "decode_hbm_frac": get(line, "decode", "roofline", "frac"),
        "decode_bf16_pool_seq_s": get(line, "decode", "bf16_state_pool", "value"),
        "decode_bf16_pool_hbm_frac": get(line, "decode", "bf16_state_pool", "roofline", "frac"),
        "long_context_decode_us_per_step": get(line, "long_context_decode", "us_per_step"),
        "long_context_decode_one_launch_us_per_step": get(line, "long_context_decode",
                                                          "rows_from_page_table_us_per_step"),
        "mixed_prefill_tok_s": get(line, "configs", "mixed_prefill", "value"),
        "mixed_prefill_hbm_frac": get(line, "configs", "mixed_prefill", "roofline", "frac"),
        "mixed_prefill_tensor_frac": get(line, "configs", "mixed_prefill", "tensor", "frac"),
        "worked_example_us": get(line, "configs", "worked_example", "prefill_call_us"),
        "tiny_prefill_us": get(line, "configs", "tiny", "prefill_call_us"),
        "tiny_decode_us": get(line, "configs", "tiny", "decode_call_us"),
        "layer_step_decode_B256_us_per_layer": get(line, "layer_step", "decode_B256", "graph_us_per_layer"),
        "cpu_oracle_tok_s": get(line, "cpu_baseline", "value"),
        "cpu_cores": get(line, "cpu_baseline", "cores"),
    }


# ---------------------------------------------------------------------------
# CPU oracle (baseline / reference arm)
# ---------------------------------------------------------------------------

def _oracle_sample(n_tok):
    """Seconds the fp64 oracle takes for the first n_tok tokens of each of the
    4 long-context sequences, all 32 heads (one paged prefill call)."""
    import oracle
    from gated_deltanet_paged_gb300 import workloads

    H, S, ps = PREFILL["H"], PREFILL["S"], PREFILL["page_size"]
    gen = torch.Generator().manual_seed(1238)
    q, k, v, g, b = workloads.draw_tokens(gen, S * n_tok, H, "cpu")
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    npg = -(-n_tok // ps)
    pool = np.zeros((S * npg, H, V, K), np.float32)
    ip = np.arange(S + 1, dtype=np.int32) * npg
    pi = np.arange(S * npg, dtype=np.int32)
    lpl = np.full(S, n_tok - (npg - 1) * ps, np.int32)
    cu = np.arange(S + 1, dtype=np.int32) * n_tok
    t0 = time.perf_counter()
    oracle.chunk_gated_delta_rule_paged(bits(q), bits(k), bits(v), g.numpy(), b.numpy(), cu, pool, pi, ip, ps,
                                        lpl, SCALE)
    return time.perf_counter() - t0


def _calibrate(target_s):
    probe = 64
    dt = _oracle_sample(probe)
    return int(max(probe, min(PREFILL["L"], probe * target_s / max(dt, 1e-3))))


def _cores():
    cores = os.cpu_count() or 1
    os.environ.setdefault("OMP_NUM_THREADS", str(cores))
    return int(os.environ["OMP_NUM_THREADS"])


def cpu_baseline(target_s=15.0):
    """The oracle as it stands, on the host cores, over a bounded sample of
    the prefill workload (~target_s seconds)."""
    cores = _cores()
    n_tok = _calibrate(target_s)
    dt = _oracle_sample(n_tok)
    return {"value": PREFILL["S"] * n_tok / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": "first %d tokens of each of the 4 long-context sequences, all 32 heads (%.1f s)"
                      % (n_tok, dt)}


def run_reference(args, rank, world):
    """Reference arm: the fp64 oracle timed on the host cores, each step a
    bounded sample of the prefill workload; rank 0 only."""
    if rank != 0:
        return None
    cores = _cores()
    per_step = args.cpu_seconds / max(1, args.steps + args.warmup)
    n_tok = _calibrate(per_step)
    for _ in range(args.warmup):
        _oracle_sample(n_tok)
    times = [_oracle_sample(n_tok) for _ in range(args.steps)]
    ms = 1e3 * sum(times) / len(times)
    value = PREFILL["S"] * n_tok / (ms * 1e-3)
    sample = "first %d tokens of each of the 4 long-context sequences, all 32 heads" % n_tok
    return {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 0, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)", "impl": "reference",
        "config": prefill_config(PREFILL["L"], world),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["gdn", "reference"], default="gdn")
    ap.add_argument("--cpu-seconds", type=float, default=20.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--workload", choices=["all", "prefill", "decode", "layers", "configs"], default="all")
    ap.add_argument("--prefill-tokens", type=int, default=PREFILL["L"],
                    help="new tokens per sequence of the prefill workload (smaller only for profiling)")
    ap.add_argument("--decode-max-ctx", type=int, default=32768,
                    help="longest context of the decode batch; with --decode-pages, a smaller pool for profiling "
                         "(the decode kernels touch one or two rows per sequence at any context)")
    ap.add_argument("--decode-pages", type=int, default=DECODE["num_pages"])
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3) if args.impl == "gdn" else args.warmup
    rank, world, local_rank = launch_env()
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        line = run_gpu(args, rank, world, local_rank)
    if rank == 0 and line is not None:
        print(json.dumps(line))


if __name__ == "__main__":
    main()

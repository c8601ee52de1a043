"""Benchmark: MLA decode (absorbed form, paged latent KV cache) on GB300.

One step = one full decode call (split-KV attention kernel + LSE combine) over
the resident synthetic MTP-3 workload (B=64, H=32, q_len=4, kv_len=81920,
page 64, bf16 cache).  The KV stream (6.04 GB) is larger than L2, so no flush
is needed between timed steps; workloads that read less than four times the L2
size (plain, tiny) get L2 flushed by a 2x-L2 write before every timed step and
are timed per step with events (``--l2-flush``).  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun (N > 1) every rank decodes its own batch (weak scaling, no
collective on the data path); rank 0 prints the max-over-ranks timing.
``--impl reference`` times the CPU oracle on a bounded sample of the same
workload on this host's cores (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MLA decode µs/call, GB/s & % of roofline (B=64,H=32,q_len=4,kv=80k)"
UNIT = "us/call"
KERNEL_SRC = os.path.join(ROOT, "mla_paged_kv_02_gb300", "csrc")
SPLIT_KERNEL_FILES = ("mla_split_kv_tc.cu", "ptx_sm100.cuh", "common.cuh")


def algorithmic_bytes(inp, out_elem_bytes):
    """Every visible KV row read once, Q read once, out + lse written once."""
    e = 1 if inp.kv_fp8 else 2
    qe = 1 if inp.q_fp8 else 2
    rows = inp.batch * inp.q_len * inp.num_heads
    kv = int(inp.seq_lens.to(torch.int64).sum().item()) * 576 * e
    return kv + rows * 576 * qe + rows * (512 * out_elem_bytes + 4)


def visible_pairs(inp):
    """(row, token) pairs the causal mask lets through: sum over requests, heads and
    query rows i of L - q_len + 1 + i."""
    L = inp.seq_lens.to(torch.int64)
    q = inp.q_len
    return int((q * L - q * (q - 1) // 2).sum().item()) * inp.num_heads


def algorithmic_flops(inp):
    """2*576 (QK) + 2*512 (PV) flops per visible (row, token) pair."""
    return 2176 * visible_pairs(inp)


def needs_l2_flush(call_bytes, l2_bytes, mode="auto"):
    """Flush L2 before every timed step?  'auto': when a call reads less than four
    times the L2 size (its inputs would partly survive in L2 between steps)."""
    return mode == "on" or (mode == "auto" and call_bytes < 4 * l2_bytes)


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def kernel_source_sha():
    h = hashlib.sha256()
    for f in SPLIT_KERNEL_FILES:
        with open(os.path.join(KERNEL_SRC, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload):
    """DRAM bytes per launch of the split kernel from a committed ncu summary, if it was
    taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    ent = d.get(workload)
    if not ent or ent.get("kernel_sha") != kernel_source_sha():
        return None
    return ent.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        fd, self.path = tempfile.mkstemp(prefix="mla_bench_clocks_", suffix=".csv")
        os.close(fd)

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(world, v):
    if world == 1:
        return v
    import torch.distributed as dist

    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def cpu_baseline(inp, reqs, threads=None):
    """Time the oracle as it stands on a bounded sample (a few requests of the same
    workload) using all host cores; scale to a whole call."""
    import oracle
    from mla_paged_kv_02_gb300 import synth

    sub = synth.subset(inp, reqs)
    threads = threads or os.cpu_count() or 1
    t0 = time.perf_counter()
    oracle.decode(sub, threads=threads)
    dt = time.perf_counter() - t0
    return dt * inp.batch / len(reqs) * 1e6, threads, dt


def run_reference(args, world, rank):
    """Reference arm: the CPU oracle on a bounded sample per step (rank 0 only).

    A whole MTP-3 call takes the fp64 oracle about a minute on 16 cores, so each
    step evaluates one request of the call (1/64 of its work) and ``value`` is
    that time scaled to the whole call; ``ms_per_step`` is the time a step
    really took, so steps x ms_per_step is the wall time of the timed region."""
    if rank != 0:
        return
    from mla_paged_kv_02_gb300 import synth

    inp = synth.make_inputs("mtp3", seed=2, device="cpu" if not torch.cuda.is_available() else "cuda")
    reqs = [0]
    times, step_s = [], []
    for k in range(args.warmup + args.steps):
        us, cores, dt = cpu_baseline(inp, reqs)
        if k >= args.warmup:
            times.append(us)
            step_s.append(dt)
    v = statistics.mean(times)
    scale = inp.batch / len(reqs)
    sample = (f"1 of {inp.batch} requests (all {inp.num_heads * inp.q_len} rows x {int(inp.seq_lens[0])} "
              f"tokens) per step; value = step time x{scale:g}")
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": statistics.mean(step_s) * 1e3,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": "mtp3: B=64 H=32 q_len=4 kv_len=81920 page=64 bf16 KV, CPU oracle sample"},
            "extrapolated": {"from_sample_fraction": len(reqs) / inp.batch, "factor": scale},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def rank_seed(workload_index, rank):
    """Every rank decodes its own batch (weak scaling): distinct seeds per rank."""
    return workload_index + 1000 * rank


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default="mtp3")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the request count (smaller cases of the same kernel for ncu)")
    ap.add_argument("--force-splits", type=int, default=0, help="override the planner's split count")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--l2-flush", default="auto", choices=["auto", "on", "off"],
                    help="write a 2x-L2 buffer before every timed step (auto: when a call reads < 4x L2)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
        return

    from mla_paged_kv_02_gb300 import _lib, api, synth

    _lib.load()
    name = args.workload
    # "fp8q" is the FP8 workload with an FP8 query too (QK^T on the FP8 tensor
    # path through mla_decode_fp8); its data are the FP8 workload's draws.
    q8 = name == "fp8q"
    base = "fp8" if q8 else name
    inp = synth.make_inputs(base, seed=rank_seed(list(synth.WORKLOADS).index(base), rank), device="cuda",
                            batch=args.batch, q_fp8=q8)
    pl = api.plan_for(inp, force_splits=args.force_splits)
    ws = api.alloc_workspace(pl, "cuda")
    out, lse = api.alloc_outputs(inp)
    kvs = api.kv_scale_tensor(inp)
    qs = torch.tensor([inp.q_scale], dtype=torch.float32, device="cuda") if q8 else None
    stream = torch.cuda.current_stream()
    qn, qp = inp.q_nope.view(-1, 512), inp.q_pe.view(-1, 64)

    def call(qn_, qp_, bt_, sl_, ev=None):
        """One decode; with events, [0]-[1] brackets the split kernel and [1]-[2] the
        combine (an FP8-query call is one C call: [0]-[1] brackets both)."""
        if ev:
            ev[0].record(stream)
        if q8:
            st = _lib.decode_fp8(pl, qn_, qp_, qs, inp.kv_cache, bt_, sl_, inp.softmax_scale, kvs, out, None, lse,
                                 ws, stream)
            st2 = 0
            if ev:
                ev[1].record(stream)
        else:
            st = _lib.split_kv(pl, qn_, qp_, inp.kv_cache, bt_, sl_, inp.softmax_scale, kvs, out, lse, ws, stream)
            if ev:
                ev[1].record(stream)
            st2 = _lib.combine(pl, out, lse, ws, stream)
        if ev:
            ev[2].record(stream)
        assert st == 0 and st2 == 0, (st, st2)

    def step(ev=None):
        call(qn, qp, inp.block_table, inp.seq_lens, ev)

    # L2 hygiene: a call that reads less than four times the L2 size would find
    # part of its inputs left in L2 by the previous step, so such workloads get
    # a 2x-L2 write before each timed step and are timed per step with events
    # (the flush is outside the bracket); larger ones stream past L2.
    l2_bytes = torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size
    out_b = 4 if inp.out_fp32 else 2
    abytes = algorithmic_bytes(inp, out_b)
    flush = needs_l2_flush(abytes, l2_bytes, args.l2_flush)
    scrub = torch.empty(2 * l2_bytes // 4, dtype=torch.int32, device="cuda") if flush else None

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st, info = _lib.check_error(ws)
    assert st == 0, (st, info)

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for k in range(args.steps):
        if flush:
            scrub.fill_(k)
        step(evs[k])
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    total_ms = t_start.elapsed_time(t_end)
    split_ms = [e[0].elapsed_time(e[1]) for e in evs]
    comb_ms = [e[1].elapsed_time(e[2]) for e in evs]
    if flush:  # per-step brackets: the flush writes between them are not the decode's
        step_us = statistics.mean(e[0].elapsed_time(e[2]) for e in evs) * 1e3
    else:
        step_us = total_ms / args.steps * 1e3
    step_us = max_over_ranks(world, step_us)
    split_us = statistics.mean(split_ms) * 1e3
    comb_us = statistics.mean(comb_ms) * 1e3

    # End to end through the public C-ABI call with host buffers: per step the
    # per-call inputs (q_nope, q_pe, block_table, seq_lens) go host->device from
    # pinned memory and out + lse come back; the KV cache is resident model state.
    h_qn = qn.cpu().pin_memory()
    h_qp = qp.cpu().pin_memory()
    h_bt = inp.block_table.cpu().pin_memory()
    h_sl = inp.seq_lens.cpu().pin_memory()
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h_lse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    d_qn, d_qp = torch.empty_like(qn), torch.empty_like(qp)
    d_bt, d_sl = torch.empty_like(inp.block_table), torch.empty_like(inp.seq_lens)
    h2d = sum(t.numel() * t.element_size() for t in (h_qn, h_qp, h_bt, h_sl))
    d2h = h_out.numel() * h_out.element_size() + h_lse.numel() * h_lse.element_size()

    def decode_into(d_qn, d_qp, d_bt, d_sl, o, l):
        if q8:
            st = _lib.decode_fp8(pl, d_qn, d_qp, qs, inp.kv_cache, d_bt, d_sl, inp.softmax_scale, kvs, o, None,
                                 l, ws, stream)
        else:
            st = _lib.decode(pl, d_qn, d_qp, inp.kv_cache, d_bt, d_sl, inp.softmax_scale, kvs, o, l, ws, stream)
        assert st == 0

    def e2e_step():
        d_qn.copy_(h_qn, non_blocking=True)
        d_qp.copy_(h_qp, non_blocking=True)
        d_bt.copy_(h_bt, non_blocking=True)
        d_sl.copy_(h_sl, non_blocking=True)
        decode_into(d_qn, d_qp, d_bt, d_sl, out, lse)
        h_out.copy_(out, non_blocking=True)
        h_lse.copy_(lse, non_blocking=True)

    # Serial: every step copies its inputs in, decodes and copies its result out
    # on one stream.
    for _ in range(args.warmup):
        e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_serial_us = max_over_ranks(world, e0.elapsed_time(e1) / args.steps * 1e3)

    # Pipelined, as a serving loop runs: the same copies, every step, but on
    # two copy streams (host to device, device to host: both directions move at
    # once) with two sets of device buffers, so that step k+1's inputs go in
    # and step k's result comes out while step k decodes.  Step k waits for its
    # own inputs; a buffer set is reused only once its previous decode and
    # read-back have finished.
    copy_stream = torch.cuda.Stream()   # host to device
    back_stream = torch.cuda.Stream()   # device to host
    sets = [dict(qn=torch.empty_like(qn), qp=torch.empty_like(qp), bt=torch.empty_like(inp.block_table),
                 sl=torch.empty_like(inp.seq_lens), out=torch.empty_like(out), lse=torch.empty_like(lse),
                 h_out=torch.empty(out.shape, dtype=out.dtype).pin_memory(),
                 h_lse=torch.empty(lse.shape, dtype=lse.dtype).pin_memory(),
                 h2d=torch.cuda.Event(), done=torch.cuda.Event(), d2h=torch.cuda.Event()) for _ in range(2)]

    def issue_inputs(b):
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(b["done"])  # its previous decode has read the inputs
            for d, h in ((b["qn"], h_qn), (b["qp"], h_qp), (b["bt"], h_bt), (b["sl"], h_sl)):
                d.copy_(h, non_blocking=True)
            b["h2d"].record(copy_stream)

    def run_pipelined(n):
        issue_inputs(sets[0])
        for k in range(n):
            b = sets[k % 2]
            if k + 1 < n:
                issue_inputs(sets[(k + 1) % 2])
            stream.wait_event(b["h2d"])
            stream.wait_event(b["d2h"])  # its previous result has been read back
            decode_into(b["qn"], b["qp"], b["bt"], b["sl"], b["out"], b["lse"])
            b["done"].record(stream)
            with torch.cuda.stream(back_stream):
                back_stream.wait_event(b["done"])
                b["h_out"].copy_(b["out"], non_blocking=True)
                b["h_lse"].copy_(b["lse"], non_blocking=True)
                b["d2h"].record(back_stream)

    run_pipelined(args.warmup)
    torch.cuda.synchronize()
    barrier(world)
    p0 = torch.cuda.Event(enable_timing=True)
    p1 = torch.cuda.Event(enable_timing=True)
    p0.record(copy_stream)
    run_pipelined(args.steps)
    stream.wait_stream(copy_stream)
    stream.wait_stream(back_stream)
    p1.record(stream)
    torch.cuda.synchronize()
    e2e_us = max_over_ranks(world, p0.elapsed_time(p1) / args.steps * 1e3)
    for b in sets:  # the pipelined results are the serial ones
        assert torch.equal(b["h_out"], h_out) and torch.equal(b["h_lse"], h_lse)
    st, info = _lib.check_error(ws)
    assert st == 0, (st, info)

    hbm_peak, tc_peak, tc_sus, peak_kind = read_peaks()
    aflops = algorithmic_flops(inp)
    achieved_gbs = abytes / (split_us * 1e-6) / 1e9
    achieved_tf = aflops / (split_us * 1e-6) / 1e12
    traffic = recorded_traffic(name)
    # The binding roofline is the one with the longer floor for this workload:
    # HBM for few query rows per page, the tensor pipe for many (e.g. 256 rows).
    hbm = {"achieved": achieved_gbs, "peak": hbm_peak, "unit": "GB/s", "frac": achieved_gbs / hbm_peak}
    tc = {"achieved": achieved_tf, "peak": tc_peak, "unit": "TFLOP/s", "frac": achieved_tf / tc_peak}
    if inp.kv_fp8 and not q8:
        # f16 operands (the FP8 cache widened exactly); f16 and bf16 share the
        # nominal dense tensor rate, so the measured bf16 peak stands for both.
        tc["peak_note"] = "f16 MMA at the measured bf16 peak (same nominal rate)"
    if q8:
        # QK^T (2*576 flops per pair) runs at the FP8 rate, taken as the measured
        # bf16 peak x 2 (the nominal dense fp8/bf16 ratio); PV (2*512, f16
        # operands) at the bf16 rate.
        pairs = visible_pairs(inp)
        floor_s = 1152 * pairs / (2 * tc_peak * 1e12) + 1024 * pairs / (tc_peak * 1e12)
        eff_peak = aflops / floor_s / 1e12
        tc = {"achieved": achieved_tf, "peak": eff_peak, "unit": "TFLOP/s", "frac": achieved_tf / eff_peak,
              "peak_note": "QK at 2x measured bf16 (fp8), PV (f16) at measured bf16; timed split+combine"}
    if aflops / (tc["peak"] * 1e12) > abytes / (hbm_peak * 1e9):
        roofline = {"bound": "tensor", **tc, "traffic": traffic, "peak_source": peak_kind, "hbm": hbm}
    else:
        roofline = {"bound": "hbm", **hbm, "traffic": traffic, "peak_source": peak_kind, "tensor": tc}

    line = {
        "metric": METRIC, "value": step_us, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_us / 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None,
        "dtype": ("fp8-e4m3 Q and KV (QK on the fp8 tensor path), f16 PV, f32 accumulate" if q8 else
                  "fp8-e4m3 KV widened to f16, f16 MMA, f32 accumulate" if inp.kv_fp8 else "bf16"),
        "data": "synthetic",
        "config": {"workload": f"{name}: B={inp.batch} H={inp.num_heads} q_len={inp.q_len} "
                               f"kv_len={'x'.join(sorted(set(str(int(x)) for x in inp.seq_lens.tolist()))) if len(set(inp.seq_lens.tolist())) == 1 else 'mixed'} "
                               f"page=64 {'e4m3' if inp.kv_fp8 else 'bf16'} KV"
                               f"{', e4m3 Q' if q8 else ''}",
                   "num_kv_splits": pl.num_kv_splits, "chunk_tokens": pl.chunk_tokens,
                   "row_groups": pl.row_groups, "partial_bytes": pl.partial_bytes,
                   "l2": ("L2 flushed before every timed step (2x-L2 write), per-step events" if flush
                          else "inputs larger than L2 (no flush)"), "parallelism": f"replicas x{world}"},
        "gb_per_s": abytes * world / (step_us * 1e-6) / 1e9,
        "tflops": aflops * world / (step_us * 1e-6) / 1e12,
        "kernel_us": ({"split_kv+combine": split_us} if q8 else {"split_kv": split_us, "combine": comb_us}),
        "roofline": roofline,
        # The faster of the two ways a caller can drive the same copies and
        # decodes (overlapped wins except for launch-bound tiny steps, where
        # the cross-stream waits cost more than they hide); both are reported.
        "e2e": {"value": min(e2e_us, e2e_serial_us), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "mode": ("copies on two copy streams (one per direction), overlapping the neighbouring steps' decodes"
                         if e2e_us <= e2e_serial_us else "one stream: copy in, decode, copy out"),
                "pipelined_value": e2e_us, "serial_value": e2e_serial_us},
        "gpu_launches": args.steps * (1 + (pl.num_kv_splits > 1)),
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        nreq = min(10, inp.batch)
        us, cores, dt = cpu_baseline(inp, list(range(nreq)))
        line["cpu_baseline"] = {"value": us, "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": f"{nreq} of {inp.batch} requests ({inp.num_heads * inp.q_len} rows x "
                                          f"{int(inp.seq_lens[0])} tokens each) in {dt:.1f} s, "
                                          f"scaled x{inp.batch / nreq:g}"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()

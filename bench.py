#!/usr/bin/env python3
"""Benchmark of the barrier-free small-message AllReduce on one GB300.

Workload (tensor-parallel decode): R = 8 simulated ranks, 8192 bf16 elements
per rank (16 KB, hidden 8192, batch 1), values normal(0, 1) with seed 1, 160
AllReduce calls per simulated token (80 layers x 2), 64 tokens.  Each token's
160 calls are one CUDA graph; the 64 token graphs use distinct input and
output buffers (1.34 GB of inputs, larger than L2), and a step is one token.

Printed: ONE JSON line with the headline (microseconds per call of the
chosen protocol), the per-protocol latencies, the measured floor (empty
graph-launched kernel + one L2 flag round trip), the end-to-end number
through the public API with host buffers, the HBM roofline of the
large-message path, and the CPU oracle timed on the host.

  python bench.py [--steps K] [--warmup W] [--proto ll] [--mode serial]
  python bench.py --impl reference      # the CPU oracle as the reference arm
  torchrun ... bench.py --gpus N        # N independent replicas, max over ranks
"""
import argparse
import glob
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from barrier_free_message_gb300 import _build, inputs, sfar  # noqa: E402

METRIC = "AllReduce µs/call at R=8, 16 KB/rank bf16 (graph-chained); GB/s vs HBM peak"
WORKLOAD = "tp-decode-r8-16k"
CALLS_PER_STEP = 160
TOKENS = 64
PROTOS = ["ll", "ll128", "sentinel", "db", "baseline"]


# --------------------------------------------------------------- distributed
def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int) -> float:
    """Largest value over all ranks (every rank gets it)."""
    if world <= 1:
        return value
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self):
        self.lines = []
        self.proc = None
        self.thread = None
        try:
            uuid = str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
            self.gpu = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            self.gpu = str(torch.cuda.current_device())

    def start(self):
        cmd = ["nvidia-smi", f"--id={self.gpu}", "--query-gpu=" + ",".join(self.FIELDS),
               "--format=csv,noheader,nounits", "-lms", "50"]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.15)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=5)
        sm, smax, reasons = [], [], set()
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(self.REASONS, parts[4:]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------- helpers
def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


KERNEL_SOURCES = {"k_ll": ("k_ll.cu", "sfar_units.cuh"), "k_sentinel": ("k_sentinel.cu", "sfar_units.cuh"),
                  "k_db": ("k_db.cu",), "k_baseline": ("k_db.cu",), "k_ll128": ("k_ll128.cu",),
                  "k_tma": ("k_tma.cu",)}


def kernel_sources_hash(kernel: str) -> str:
    """Hash of the files that make up one kernel (its own sources and the shared headers)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "barrier_free_message_gb300", "csrc")
    for name in (*KERNEL_SOURCES.get(kernel, ()), "sfar_prims.cuh", "sfar_internal.h"):
        p = os.path.join(csrc, name)
        if os.path.isfile(p):
            with open(p, "rb") as f:
                h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources; otherwise None."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            t = json.load(f)
        e = t.get(kernel)
        if e and e.get("sources") == kernel_sources_hash(kernel):
            return e.get("dram_bytes_per_launch")
    except Exception:
        pass
    return None


def gen_calls(w, calls):
    x = torch.empty((calls, w.R, w.n), dtype=torch.bfloat16 if w.dtype == "bf16" else torch.float32)
    for c in range(calls):
        x[c] = inputs.draw_workload_call(w, c)
    return x


def capture_token_graphs(h, x_dev, out_dev, proto, tokens):
    calls, R, n = x_dev.shape
    graphs = []
    for t in range(tokens):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for c in range(t * CALLS_PER_STEP, (t + 1) * CALLS_PER_STEP):
                code = sfar.sfar_allreduce(h.h, [x_dev[c, r].data_ptr() for r in range(R)],
                                           [out_dev[c, r].data_ptr() for r in range(R)], n, proto)
                if code != sfar.SFAR_OK:
                    raise sfar.SfarError(code, "sfar_allreduce during capture")
        graphs.append(g)
    return graphs


def time_graphs(graphs, steps, warmup, world, sampler=None):
    stream = torch.cuda.current_stream()
    for i in range(warmup):
        graphs[i % len(graphs)].replay()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(steps):
        graphs[(warmup + i) % len(graphs)].replay()
    end.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    barrier(world)
    ms = start.elapsed_time(end)
    return max_over_ranks(ms, world), clocks


def check_status(h, what):
    code, f = sfar.sfar_status_get(h.h)
    if code != sfar.SFAR_OK:
        raise RuntimeError(f"{what}: device status {sfar.strerror(code)} (rank {f.rank} cta {f.cta} peer {f.peer} "
                           f"epoch {f.epoch} where {sfar.WAIT_NAMES.get(f.where, f.where)})")


def floor_probe():
    """Empty graph-launched kernel + one L2 flag round trip, in microseconds."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(CALLS_PER_STEP):
            assert sfar.sfar_probe_empty() == sfar.SFAR_OK
    for _ in range(5):
        g.replay()
    torch.cuda.synchronize()
    reps = 50
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(reps):
        g.replay()
    e.record()
    torch.cuda.synchronize()
    empty_us = s.elapsed_time(e) * 1000.0 / (reps * CALLS_PER_STEP)
    flags = torch.zeros(64, dtype=torch.int32, device="cuda")
    out = torch.zeros(3, dtype=torch.int64, device="cuda")
    trips = 5000
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    # every partner CTA (one CTA per SM): which SMs the two CTAs land on (same
    # die or not) sets the round trip, and the AllReduce's CTAs cover every SM,
    # so the floor takes the slowest pair (each pair the best of two runs)
    partners = list(range(1, sms))

    def rtt(relaxed, partner):
        best = None
        for _ in range(2):
            assert sfar.sfar_probe_pingpong(flags.data_ptr(), trips, out.data_ptr(), relaxed, partner) == sfar.SFAR_OK
            torch.cuda.synchronize()
            v = out.cpu().tolist()
            if v[0] < 0:
                raise RuntimeError("ping-pong probe timed out")
            us = v[0] / trips / 1000.0
            best = (us, v[1], v[2]) if best is None or us < best[0] else best
        return best

    acq = [rtt(False, p) for p in partners]
    rel = [rtt(True, p) for p in partners]
    a_us = sorted(x[0] for x in acq)
    r_us = sorted(x[0] for x in rel)
    slow = max(acq)
    return {"empty_kernel_us": empty_us, "flag_rtt_us": a_us[-1], "floor_us": empty_us + a_us[-1],
            "flag_rtt_min_us": a_us[0], "flag_rtt_median_us": a_us[len(a_us) // 2],
            "flag_rtt_p90_us": a_us[int(0.9 * (len(a_us) - 1))],
            "relaxed_flag_rtt_us": r_us[-1], "relaxed_flag_rtt_min_us": r_us[0],
            "slowest_pair_sm": [slow[1], slow[2]], "pairs": len(partners)}


def spot_check(out_dev, x_host, calls):
    """Bit-exact comparison of a few calls with the CPU oracle."""
    import oracle
    for c in calls:
        want = oracle.allreduce(inputs.to_bits(x_host[c]))
        got = inputs.to_bits(out_dev[c].cpu())
        if not np.array_equal(got, want):
            return False
    return True


def replayed_tokens(tokens, warmup, steps):
    """Token graphs that the warm-up and timed replays ran (replay i runs token i % tokens)."""
    return sorted({i % tokens for i in range(warmup + steps)})


def oracle_rows(x_host, call_ids, threads):
    """The oracle's result of each call in call_ids: [len(call_ids), n] bits
    (every rank receives the same row), computed with the oracle's
    multithreaded variant (the same bits as one thread)."""
    import oracle
    xs = x_host[call_ids]
    m, R, n = xs.shape
    flat = inputs.to_bits(xs.transpose(0, 1).reshape(R, m * n))
    return oracle.allreduce(flat, threads=threads)[0].reshape(m, n)


def _as_int(t):
    """bf16 / fp32 data as int16 / int32 bit patterns (integer tensors unchanged)."""
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16)
    if t.dtype == torch.float32:
        return t.view(torch.int32)
    return t


def device_mismatches(out_dev, call_ids, exp_dev, block=1024):
    """Calls among call_ids whose output differs from the oracle's row
    (exp_dev, [len(call_ids), n] on the device) on any rank: compared on the
    device, block by block."""
    bad = 0
    ids = torch.as_tensor(call_ids, device=out_dev.device)
    for i in range(0, len(call_ids), block):
        got = _as_int(out_dev)[ids[i:i + block]]
        eq = (got == _as_int(exp_dev[i:i + block])[:, None, :]).all(dim=2).all(dim=1)
        bad += int((~eq).sum())
    return bad


def admissible_check(out_dev, x_host, calls):
    """The order-free (atomic) protocol: every rank equal and every element of
    a few calls inside the oracle's admissible interval."""
    from oracle import atomic
    for c in calls:
        got = inputs.to_bits(out_dev[c].cpu())
        if not all(np.array_equal(got[r], got[0]) for r in range(1, got.shape[0])):
            return False
        if not atomic.check(inputs.to_bits(x_host[c]), got[0]).all():
            return False
    return True


def large_message_roofline(peak_gbs, R=8, mb=64, dtype="bf16", reps=10, check=True):
    """HBM roofline of the two-shot TMA path: 2*R*S bytes per call.  Two
    input/output buffer sets (2 * 2 * R * S bytes, above L2 from 4 MB per rank
    at R >= 4) alternate inside one CUDA graph (2 calls, up to 16 for small
    messages so that the gap between graph replays is spread thin), so the
    timing holds no host launch cost; every element of the last call of each
    set is then compared with the oracle."""
    es = 2 if dtype == "bf16" else 4
    n = (mb << 20) // es
    h = sfar.Sfar(R, mb << 20, dtype)
    sets = []
    for s in range(2):
        ins = inputs.draw_device(4, s, R, n, "normal", 1.0, dtype)
        outs = [torch.empty_like(t) for t in ins]
        sets.append((ins, outs))
    for i in range(2):
        h.allreduce(*sets[i], "twoshot_tma")
    torch.cuda.synchronize()
    per_graph = 2 * max(1, min(8, 64 // mb))          # small messages: more calls per graph replay
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(per_graph):
            h.allreduce(*sets[i % 2], "twoshot_tma")
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    s_ev, e_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s_ev.record()
    for _ in range(reps):
        g.replay()
    e_ev.record()
    torch.cuda.synchronize()
    check_status(h, "twoshot_tma")
    ms = s_ev.elapsed_time(e_ev) / (per_graph * reps)
    ok = None
    if check:
        import oracle
        ok = True
        for ins, outs in sets:
            xb = np.stack([inputs.to_bits(t.cpu()) for t in ins])
            want = oracle.allreduce(xb, threads=os.cpu_count() or 1)[0]
            exp = torch.from_numpy(want.view(np.int16) if es == 2 else want.view(np.int32)).cuda()
            ok = ok and all(bool(torch.equal(_as_int(o), exp)) for o in outs)
            del xb, want, exp
    k, _ = h.launch(n, "twoshot_tma")
    h.close()
    del sets, g
    byts = 2 * R * (mb << 20)
    gbs = byts / (ms * 1e-3) / 1e9
    return {"bound": "hbm", "kernel": "k_tma", "workload": f"R={R}, {mb} MB/rank {dtype}, two-shot TMA",
            "achieved": round(gbs, 1), "peak": peak_gbs, "unit": "GB/s", "frac": round(gbs / peak_gbs, 4),
            "us_per_call": round(ms * 1000, 2), "algorithmic_bytes": byts, "ctas_per_rank": k,
            "traffic": profiled_traffic("k_tma"), "bit_exact": ok,
            "timing": "CUDA graph of %d calls alternating two buffer sets, 3 warm-up + %d timed replays"
                      % (per_graph, reps)}


def oracle_cpu_time(x_host, budget_s=10.0, calls_per_step=None, threads=1):
    """The oracle as it stands on a bounded sample of calls: single-threaded,
    or with each call's elements split over `threads` threads (its
    multithreaded variant, the same bits)."""
    import oracle
    xs = [inputs.to_bits(x_host[c]) for c in range(min(len(x_host), 2048))]
    oracle.allreduce(xs[0], threads=threads)
    done, t0 = 0, time.perf_counter()
    while True:
        oracle.allreduce(xs[done % len(xs)], threads=threads)
        done += 1
        if calls_per_step is not None:
            if done >= calls_per_step:
                break
        elif time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return dt / done * 1e6, done, dt


# ----------------------------------------------------------------- suites
ALL = PROTOS + ["twoshot", "twoshot_sent", "twoshot_tma"]


def _time_chain(h, x_dev, out_dev, proto, reps=40, warm=3):
    """Capture one graph of all calls in x_dev and time `reps` replays (µs per call)."""
    calls, R, n = x_dev.shape
    h.allreduce([x_dev[0, r] for r in range(R)], [out_dev[0, r] for r in range(R)], proto)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for c in range(calls):
            code = sfar.sfar_allreduce(h.h, [x_dev[c, r].data_ptr() for r in range(R)],
                                       [out_dev[c, r].data_ptr() for r in range(R)], n, proto)
            if code != sfar.SFAR_OK:
                raise sfar.SfarError(code, "capture")
    for _ in range(warm):
        g.replay()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(reps):
        g.replay()
    e.record()
    torch.cuda.synchronize()
    check_status(h, proto)
    return s.elapsed_time(e) * 1000.0 / (reps * calls)


def _oracle_us(fn, budget_s=2.0):
    """The oracle (CPU, one thread) timed on one call of a suite's workload:
    µs per call, repeated while under the budget."""
    t0 = time.perf_counter()
    n = 0
    while True:
        fn()
        n += 1
        if time.perf_counter() - t0 > budget_s or n >= 100:
            break
    return round((time.perf_counter() - t0) * 1e6 / n, 1)


def _time_calls(h, calls, steps, reps=40, warm=3):
    """One graph of `calls` iterations of the call sequence `steps` (each a
    function of the call index returning a status); µs per iteration."""
    for f in steps:
        code = f(0)
        if code != sfar.SFAR_OK:
            raise sfar.SfarError(code, "warm-up")
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for c in range(calls):
            for f in steps:
                code = f(c)
                if code != sfar.SFAR_OK:
                    raise sfar.SfarError(code, "capture")
    for _ in range(warm):
        g.replay()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(reps):
        g.replay()
    e.record()
    torch.cuda.synchronize()
    check_status(h, "suite")
    return s.elapsed_time(e) * 1000.0 / (reps * calls)


def run_suite(args):
    """Sweeps printed as JSON lines: the latency curve of every protocol over
    message sizes (R = 4, 8; both launch modes), the bandwidth of the TMA path
    (R = 2..16, bf16 and fp32, 4-256 MB per rank), the cost of the barriers
    against the rank count (BASELINE vs DB vs LL vs sentinel, 16 KB per rank,
    R = 2..16), the atomic-accumulation two-shot against the two-shot,
    LL128 and LL protocols (R = 4, 8, 16 over message sizes), the fused
    AllReduce + residual add + RMSNorm against the two-kernel pipeline, and
    a synthetic tensor-parallel decode step (row-parallel projections and
    their AllReduces) under three launch configurations."""
    _build.build()
    l2 = torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size
    # the latency floor of this box (empty graph kernel + slowest flag round
    # trip), measured once: the roofline of the latency-bound suites
    floor_us = floor_probe()["floor_us"] if {"atomic", "fused"} & set(args.suite.split(",")) else None
    if floor_us is not None:
        print(json.dumps({"suite": "floor", "floor_us": round(floor_us, 3)}), flush=True)
    if "latency" in args.suite:
        for R in (4, 8, 16):
            if args.suite_r and R != args.suite_r:
                continue
            h = sfar.Sfar(R, 1 << 20, "bf16")
            for b in inputs.SWEEP_BYTES:
                if args.suite_bytes and b != args.suite_bytes:
                    continue
                n, calls = b // 2, 32
                x = torch.stack([inputs.draw(2, c, R, n, "uniform", 1.0, "bf16") for c in range(calls)])
                xd = x.cuda()
                od = torch.empty_like(xd)
                for mode in ("serial", "overlap"):
                    h.set_mode(mode)
                    for proto in (args.suite_protos.split(",") if args.suite_protos else ALL):
                        us = _time_chain(h, xd, od, proto)
                        k, t = h.launch(n, proto)
                        print(json.dumps({"suite": "latency", "R": R, "bytes": b, "mode": mode, "proto": proto,
                                          "us": round(us, 3), "ctas_per_rank": k, "threads": t,
                                          "l2_resident": 2 * calls * R * b < l2,
                                          "bit_exact_sample": spot_check(od, x, [0, calls - 1])}), flush=True)
                del xd, od
            h.close()
    if "bandwidth" in args.suite:
        peaks, _ = measured_peaks()
        for dtype in ("bf16", "fp32"):
            for R in (2, 4, 8, 16):
                if args.suite_r and R != args.suite_r:
                    continue
                for mb in (b >> 20 for b in inputs.BANDWIDTH_BYTES):
                    d = large_message_roofline(float(peaks["hbm_gbs"]), R=R, mb=mb, dtype=dtype)
                    d.update({"suite": "bandwidth", "R": R, "mb": mb, "dtype": dtype})
                    print(json.dumps(d), flush=True)
                    torch.cuda.empty_cache()
    if "barriers" in args.suite:
        n, calls = 8192, 160
        for R in (2, 3, 4, 6, 8, 12, 16):
            x = torch.stack([inputs.draw(1, c, R, n, "normal", 1.0, "bf16") for c in range(calls)])
            xd = x.cuda()
            od = torch.empty_like(xd)
            h = sfar.Sfar(R, 2 * n, "bf16")
            row = {"suite": "barriers", "R": R, "bytes": 2 * n}
            for proto in ("baseline", "db", "ll", "sentinel"):
                row[proto] = round(_time_chain(h, xd, od, proto), 3)
                row[proto + "_exact"] = spot_check(od, x, [0, calls - 1])
            row["two_barriers_minus_ll"] = round(row["baseline"] - row["ll"], 3)
            row["bottom_barrier"] = round(row["baseline"] - row["db"], 3)
            print(json.dumps(row), flush=True)
            h.close()
    if "fused" in args.suite:
        # AllReduce + residual add + RMSNorm in one kernel against the two-kernel
        # pipeline (LL AllReduce, then the normalisation kernel)
        import oracle
        for R, rows, hidden in ((8, 1, 8192), (8, 64, 7168), (4, 1, 8192), (16, 1, 8192), (8, 4, 8192),
                                (8, 8, 8192), (8, 16, 7168), (16, 64, 7168)):
            if (args.suite_r and R != args.suite_r) or (args.suite_rows and rows != args.suite_rows):
                continue
            calls, eps = 32, 1e-5
            n = rows * hidden
            x = torch.stack([inputs.draw(6, c, R, n, "normal", 1.0, "bf16") for c in range(calls)])
            res = torch.stack([inputs.draw(7, c, R, n, "normal", 2.0, "bf16") for c in range(calls)])
            w = inputs.draw(8, 0, 1, hidden, "normal", 1.0, "bf16")[0]
            xd, rd, wd = x.cuda(), res.cuda(), w.cuda()
            od, zd, ad = torch.empty_like(xd), torch.empty_like(xd), torch.empty_like(xd)
            h = sfar.Sfar(R, 2 * n, "bf16")
            h.set_mode(args.mode)
            P = lambda t, c: [t[c, r].data_ptr() for r in range(R)]

            def fused(c):
                return sfar.sfar_allreduce_add_rmsnorm(h.h, P(xd, c), P(rd, c), wd.data_ptr(), P(od, c), P(zd, c),
                                                       rows, hidden, eps)

            def allreduce(c):
                return sfar.sfar_allreduce(h.h, P(xd, c), P(ad, c), n, "ll")

            def norm(c):
                return sfar.sfar_add_rmsnorm(h.h, P(ad, c), P(rd, c), wd.data_ptr(), P(od, c), P(zd, c), rows,
                                             hidden, eps)

            row = {"suite": "fused", "R": R, "rows": rows, "hidden": hidden, "bytes_per_rank": 2 * n}
            row["fused_path"] = {1: "oneshot", 2: "twoshot"}[sfar.sfar_test_query_fused_path(h.h, rows, hidden)[1]]
            for path in ("oneshot", "twoshot"):          # each kernel forced, where the shape allows it
                sfar.sfar_test_set_fused_path(h.h, path)
                if sfar.sfar_test_query_fused_path(h.h, rows, hidden) == (sfar.SFAR_OK, 1 if path == "oneshot" else 2):
                    row[f"fused_{path}_us"] = round(_time_calls(h, calls, [fused]), 3)
            sfar.sfar_test_set_fused_path(h.h, "auto")
            row["fused_us"] = round(_time_calls(h, calls, [fused]), 3)
            ok = True
            for c in (0, calls - 1):
                wy, wz = oracle.add_rmsnorm(inputs.to_bits(x[c]), inputs.to_bits(res[c]),
                                            inputs.to_bits(w[None, :])[0], eps, hidden)
                ok = ok and np.array_equal(inputs.to_bits(od[c].cpu()), wy) and \
                    np.array_equal(inputs.to_bits(zd[c].cpu()), wz)
            row["fused_bit_exact_sample"] = bool(ok)
            row["unfused_us"] = round(_time_calls(h, calls, [allreduce, norm]), 3)
            row["allreduce_ll_us"] = round(_time_calls(h, calls, [allreduce]), 3)
            row["norm_alone_us"] = round(_time_calls(h, calls, [norm]), 3)
            row["saved_us"] = round(row["unfused_us"] - row["fused_us"], 3)
            row["fused_vs_floor"] = round(row["fused_us"] / floor_us, 3)
            xb, rb, wb = inputs.to_bits(x[0]), inputs.to_bits(res[0]), inputs.to_bits(w[None, :])[0]
            row["oracle_us"] = _oracle_us(lambda: oracle.add_rmsnorm(xb, rb, wb, eps, hidden))
            print(json.dumps(row), flush=True)
            h.close()
            del xd, rd, od, zd, ad
    if "decode" in args.suite:
        # a synthetic tensor-parallel decode step: 80 layers x (attention output
        # projection, MLP down projection), each a row-parallel projection of
        # every rank followed by the AllReduce of the partial sums (fused with
        # the residual add + RMSNorm, or plain LL); random bf16 weights of
        # 4 distinct layers (2.4 GB, far above L2) cycled over the 80
        import oracle
        peaks, _ = measured_peaks()
        hbm = float(peaks["hbm_gbs"])
        R, h, layers, distinct, eps, nx = 8, 8192, args.decode_layers, 4, 1e-5, 8
        ks = (8192 // R, 28672 // R)
        g = torch.Generator(device="cuda").manual_seed(90)
        W = [[[(torch.randn(k, h, generator=g, device="cuda") * 0.02).to(torch.bfloat16) for _ in range(R)]
              for k in ks] for _ in range(distinct)]
        X = [[[torch.randn(k, generator=g, device="cuda").to(torch.bfloat16) for _ in range(R)] for _ in range(nx)]
             for k in ks]
        calls = 2 * layers
        part = [[torch.empty(h, dtype=torch.bfloat16, device="cuda") for _ in range(R)] for _ in range(calls)]
        out = [[torch.empty(h, dtype=torch.bfloat16, device="cuda") for _ in range(R)] for _ in range(calls)]
        res = [torch.randn(h, generator=g, device="cuda").to(torch.bfloat16) for _ in range(R)]
        wn = torch.randn(h, generator=g, device="cuda").to(torch.bfloat16)
        # the oracle on one attention-output and one down projection of the
        # workload (plus their AllReduces), per projection + AllReduce
        xo = [np.stack([inputs.to_bits(t.cpu()) for t in X[kind][0]]) for kind in range(2)]
        wo = [np.stack([inputs.to_bits(t.cpu()) for t in W[0][kind]]) for kind in range(2)]
        oracle_us = round(sum(_oracle_us(lambda kind=kind: oracle.allreduce(oracle.gemv(xo[kind], wo[kind])),
                                         budget_s=0.5) for kind in range(2)) / 2, 1)
        del xo, wo
        hd = sfar.Sfar(R, 2 * h, "bf16")          # the AllReduces
        hg = sfar.Sfar(R, 2 * h, "bf16")          # the projections (own launch mode)
        P = lambda ts: [t.data_ptr() for t in ts]
        wbytes = layers * R * sum(ks) * h * 2
        # (projection launch, AllReduce launch, prefetch rows, streams): "serial" =
        # as a programmatic dependent of the kernel before it; two streams = the
        # page's pattern (section three): the projection on a compute stream,
        # the AllReduce on a communication stream, each waiting for the other's
        # event
        configs = (("plain", "plain", 0, 1), ("serial", "serial", 0, 1), ("serial", "serial", 128, 1),
                   ("serial", "plain", 128, 1), ("plain", "plain", 0, 2))
        comm = torch.cuda.Stream()
        for ar in ("fused", "ll"):
            for gmode, amode, prefetch, nstreams in configs:
                hd.set_mode(amode)
                hg.set_mode(gmode)

                def gemv_call(c, st=None):
                    kind = c % 2
                    return sfar.sfar_rowpar_gemv(hg.h, P(X[kind][(c // 2) % nx]), P(W[(c // 2) % distinct][kind]),
                                                 P(part[c]), ks[kind], h, prefetch, st)

                def ar_call(c, st=None):
                    if ar == "fused":
                        return sfar.sfar_allreduce_add_rmsnorm(hd.h, P(part[c]), P(res), wn.data_ptr(), P(out[c]),
                                                               P(res), 1, h, eps, st)
                    return sfar.sfar_allreduce(hd.h, P(part[c]), P(out[c]), h, "ll", st)

                for f in (gemv_call, ar_call):
                    assert f(0) == sfar.SFAR_OK
                torch.cuda.synchronize()
                graph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(graph):
                    cap = torch.cuda.current_stream()
                    for c in range(calls):
                        if nstreams == 1:
                            codes = (gemv_call(c), ar_call(c))
                        else:
                            g_done = torch.cuda.Event()
                            code_g = gemv_call(c, cap.cuda_stream)
                            g_done.record(cap)
                            comm.wait_event(g_done)
                            code_a = ar_call(c, comm.cuda_stream)
                            a_done = torch.cuda.Event()
                            a_done.record(comm)
                            cap.wait_event(a_done)
                            codes = (code_g, code_a)
                        for code in codes:
                            if code != sfar.SFAR_OK:
                                raise sfar.SfarError(code, "decode capture")
                for _ in range(2):
                    graph.replay()
                torch.cuda.synchronize()
                reps = 10
                t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                t0.record()
                for _ in range(reps):
                    graph.replay()
                t1.record()
                torch.cuda.synchronize()
                check_status(hd, "decode")
                us_token = t0.elapsed_time(t1) * 1000.0 / reps
                # parity sample: call 1 (an MLP down projection) and, for LL, its AllReduce
                xs1 = np.stack([inputs.to_bits(t.cpu()) for t in X[1][0]])
                w1 = np.stack([inputs.to_bits(t.cpu()) for t in W[0][1]])
                got = np.stack([inputs.to_bits(t.cpu()) for t in part[1]])
                ok = bool(np.array_equal(got, oracle.gemv(xs1, w1)))
                if ar == "ll":
                    ok = ok and bool(np.array_equal(np.stack([inputs.to_bits(t.cpu()) for t in out[1]]),
                                                    oracle.allreduce(got)))
                print(json.dumps({"suite": "decode", "ar": ar, "projection_launch": gmode, "allreduce_launch": amode,
                                  "prefetch_rows": prefetch, "streams": nstreams, "R": R,
                                  "hidden": h, "layers": layers, "calls_per_token": calls,
                                  "us_per_token": round(us_token, 1),
                                  "us_per_projection_and_allreduce": round(us_token / calls, 3),
                                  "weight_bytes_per_token": wbytes,
                                  "weight_gbs": round(wbytes / us_token / 1e3, 1),
                                  "frac_of_measured_hbm": round(wbytes / us_token / 1e3 / hbm, 4),
                                  "bit_exact_sample": ok,
                                  "oracle_us_per_projection_and_allreduce": oracle_us}), flush=True)
                del graph
        hd.close()
        hg.close()
    if "atomic" in args.suite:
        # the atomic-accumulation two-shot against the flag-line protocols
        for R in (4, 8, 16):
            if args.suite_r and R != args.suite_r:
                continue
            h = sfar.Sfar(R, 1 << 20, "bf16")
            for b in inputs.SWEEP_BYTES:
                if args.suite_bytes and b != args.suite_bytes:
                    continue
                n, calls = b // 2, 32
                x = torch.stack([inputs.draw(5, c, R, n, "normal", 1.0, "bf16") for c in range(calls)])
                xd = x.cuda()
                od = torch.empty_like(xd)
                row = {"suite": "atomic", "R": R, "bytes": b}
                for proto in ("ll128_atomic", "twoshot", "ll128", "ll"):
                    row[proto] = round(_time_chain(h, xd, od, proto), 3)
                    row[proto + "_ok"] = (admissible_check(od, x, [0, calls - 1]) if proto == "ll128_atomic"
                                          else spot_check(od, x, [0, calls - 1]))
                k, t = h.launch(n, "ll128_atomic")
                row["atomic_ctas_per_rank"], row["atomic_threads"] = k, t
                row["atomic_vs_floor"] = round(row["ll128_atomic"] / floor_us, 3)
                from oracle import atomic
                xb, ob = inputs.to_bits(x[0]), inputs.to_bits(od[0, 0].cpu())
                row["oracle_us"] = _oracle_us(lambda: atomic.check(xb, ob))   # the admissible interval of one call
                print(json.dumps(row), flush=True)
                del xd, od
            h.close()


# ----------------------------------------------------------------- arms
def workload_config(args, tokens):
    """The `config` object of the JSON line: the workload only, the same in
    both arms (launch details go under `launch`)."""
    w = inputs.WORKLOADS[WORKLOAD]
    return {"workload": WORKLOAD, "R": w.R, "n": w.n, "bytes_per_rank": w.bytes_per_rank, "io_dtype": w.dtype,
            "dist": f"{w.dist}(0,{w.sigma:g}) seed {w.seed}", "calls_per_step": CALLS_PER_STEP, "tokens": tokens,
            "l2": "inputs larger than L2: %d token buffers of %d calls (%.2f GB), cycled"
                  % (tokens, CALLS_PER_STEP, tokens * CALLS_PER_STEP * w.R * w.bytes_per_rank / 1e9),
            "parallelism": f"replicas x{args.gpus}"}


def run_reference(args, world, rank):
    if rank != 0:
        return
    import oracle  # noqa: F401
    from oracle.build import build_oracle
    build_oracle()
    w = inputs.WORKLOADS[WORKLOAD]
    x = gen_calls(w, 512)
    for _ in range(args.warmup):
        oracle_cpu_time(x, calls_per_step=CALLS_PER_STEP)
    t0 = time.perf_counter()
    total_calls = 0
    for _ in range(args.steps):
        _, n_calls, _ = oracle_cpu_time(x, calls_per_step=CALLS_PER_STEP)
        total_calls += n_calls
    dt = time.perf_counter() - t0
    us = dt / total_calls * 1e6
    line = {"impl": "reference", "metric": METRIC, "value": round(us, 3), "unit": "us/call", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3 / args.steps, 3),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": workload_config(args, args.tokens),
            "cpu_baseline": {"value": round(us, 3), "unit": "us/call", "cores": 1, "kind": "oracle",
                             "sample": f"{args.steps} steps x {CALLS_PER_STEP} calls of R=8 x 8192 bf16, "
                                       f"cycling over 512 generated calls"},
            "e2e": {"value": round(us, 3), "unit": "us/call", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def _graph_of_calls(h, x_dev, out_dev, proto):
    calls, R, n = x_dev.shape
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for c in range(calls):
            code = sfar.sfar_allreduce(h.h, [x_dev[c, r].data_ptr() for r in range(R)],
                                       [out_dev[c, r].data_ptr() for r in range(R)], n, proto)
            if code != sfar.SFAR_OK:
                raise sfar.SfarError(code, "capture")
    return g


def _time_graph(g, reps, warm=3):
    for _ in range(warm):
        g.replay()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(reps):
        g.replay()
    e.record()
    torch.cuda.synchronize()
    return s.elapsed_time(e) * 1000.0 / reps        # µs per replay


def other_configs():
    """The two other workloads that run on the AllReduce alone: R = 4 at 8 KB
    per rank (LL, 100 calls with inputs redrawn per call), and batched decode,
    R = 8 at 896 KB per rank (two-shot, 64 calls, with and without a straggler
    rank that spins 0-20 µs before its sends, rotating over the ranks).  Each
    is one CUDA graph of all its calls; every call of the last replay is
    compared bit for bit with the oracle."""
    import oracle
    res = {}
    threads = os.cpu_count() or 1

    # small: R = 4, 4096 bf16 (8 KB), uniform, seed 0, 100 calls
    w = inputs.WORKLOADS["small-r4-8k"]
    x = gen_calls(w, w.calls)
    exp = torch.from_numpy(oracle_rows(x, list(range(w.calls)), threads).view(np.int16)).cuda()
    xd = x.cuda()
    od = torch.empty_like(xd)
    h = sfar.Sfar(w.R, w.bytes_per_rank, w.dtype)
    h.allreduce([xd[0, r] for r in range(w.R)], [od[0, r] for r in range(w.R)], "ll")
    torch.cuda.synchronize()
    g = _graph_of_calls(h, xd, od, "ll")
    od.view(torch.int16).fill_(-1)
    us = _time_graph(g, reps=50) / w.calls
    check_status(h, "small ll")
    bad = device_mismatches(od, list(range(w.calls)), exp)
    xb = [inputs.to_bits(x[c]) for c in range(w.calls)]
    t0 = time.perf_counter()
    for c in range(w.calls):
        oracle.allreduce(xb[c])
    oracle_ms = (time.perf_counter() - t0) * 1e3
    res[w.name] = {"proto": "ll", "R": w.R, "bytes_per_rank": w.bytes_per_rank, "calls": w.calls,
                   "us_per_call": round(us, 3), "bit_exact": bad == 0, "calls_checked": w.calls,
                   "l2_resident": True, "oracle_ms_for_all_calls": round(oracle_ms, 2),
                   "oracle_cores": 1}
    h.close()
    del g, xd, od, exp

    # batched decode: R = 8, 64 x 7168 bf16 (896 KB), normal(0, 0.5), seed 3, 64 calls
    w = inputs.WORKLOADS["batched-decode-r8-896k"]
    x = gen_calls(w, w.calls)
    exp = torch.from_numpy(oracle_rows(x, list(range(w.calls)), threads).view(np.int16)).cuda()
    xd = x.cuda()
    od = torch.empty_like(xd)
    row = {"R": w.R, "bytes_per_rank": w.bytes_per_rank, "calls": w.calls, "l2_resident": False,
           "us_per_call": {}, "bit_exact": {}}
    for proto in sfar.EXACT_PROTOS:
        h = sfar.Sfar(w.R, w.bytes_per_rank, w.dtype)
        h.allreduce([xd[0, r] for r in range(w.R)], [od[0, r] for r in range(w.R)], proto)
        torch.cuda.synchronize()
        g = _graph_of_calls(h, xd, od, proto)
        od.view(torch.int16).fill_(-1)
        row["us_per_call"][proto] = round(_time_graph(g, reps=20) / w.calls, 3)
        check_status(h, proto)
        row["bit_exact"][proto] = device_mismatches(od, list(range(w.calls)), exp) == 0
        h.close()
        del g
    # a straggler: rank (call mod 8) spins U[0, 20] µs (seed 3) before its sends
    gen = torch.Generator().manual_seed(w.seed)
    delays = torch.randint(0, 20001, (w.calls,), generator=gen, dtype=torch.int64).to(torch.int32).cuda()
    row["straggler"] = {"rank": "call mod 8", "delay_us": "uniform integer ns in [0, 20000], seed 3",
                        "mean_delay_us": round(float(delays.double().mean()) / 1e3, 3), "us_per_call": {},
                        "bit_exact": {}}
    for proto in ("twoshot", "twoshot_sent", "twoshot_tma"):
        h = sfar.Sfar(w.R, w.bytes_per_rank, w.dtype)
        assert sfar.sfar_test_set_straggler(h.h, delays.data_ptr(), w.calls, -1, 0) == sfar.SFAR_OK
        h.allreduce([xd[0, r] for r in range(w.R)], [od[0, r] for r in range(w.R)], proto)
        torch.cuda.synchronize()
        g = _graph_of_calls(h, xd, od, proto)
        od.view(torch.int16).fill_(-1)
        row["straggler"]["us_per_call"][proto] = round(_time_graph(g, reps=10) / w.calls, 3)
        check_status(h, proto + " straggler")
        row["straggler"]["bit_exact"][proto] = device_mismatches(od, list(range(w.calls)), exp) == 0
        h.close()
        del g
    res[w.name] = row
    del xd, od, exp
    return res


def run_ours(args, world, rank):
    _build.build()
    sfar.lib()
    w = inputs.WORKLOADS[WORKLOAD]
    tokens = args.tokens
    calls = tokens * CALLS_PER_STEP
    peaks, peak_kind = measured_peaks()
    hbm_peak = float(peaks.get("hbm_gbs", 6800.0))
    if args.large_only:
        large = large_message_roofline(hbm_peak, R=args.large_r, mb=args.large_mb, dtype=args.large_dtype)
        if rank == 0:
            print(json.dumps({"roofline_large": large}), flush=True)
        return

    x_host = gen_calls(w, calls).pin_memory()
    x_dev = x_host.cuda()
    out_dev = torch.empty_like(x_dev)
    out_host = torch.empty_like(x_host).pin_memory()
    e2e_steps = 0 if args.no_e2e else min(args.steps, 4 * tokens)

    # the oracle's rows of every call that the replays and the end-to-end
    # loop compute (the replays run tokens (warm-up + i) % tokens)
    replay = replayed_tokens(tokens, args.warmup, args.steps)
    e2e_tokens = sorted({i % tokens for i in range(e2e_steps)})
    check_tokens = sorted(set(replay) | set(e2e_tokens))
    pos = {t: i for i, t in enumerate(check_tokens)}
    check_ids = [t * CALLS_PER_STEP + c for t in check_tokens for c in range(CALLS_PER_STEP)]
    t_or = time.perf_counter()
    exp_rows = oracle_rows(x_host, check_ids, os.cpu_count() or 1)
    oracle_check_s = time.perf_counter() - t_or
    exp_dev = torch.from_numpy(exp_rows.view(np.int16)).cuda()
    replay_ids = [t * CALLS_PER_STEP + c for t in replay for c in range(CALLS_PER_STEP)]
    replay_rows = torch.as_tensor([pos[t] * CALLS_PER_STEP + c for t in replay for c in range(CALLS_PER_STEP)],
                                  device="cuda")

    h = sfar.Sfar(w.R, w.bytes_per_rank, w.dtype)
    h.set_mode(args.mode)
    if args.geometry:
        kk, tt = (int(v) for v in args.geometry.split(","))
        assert sfar.sfar_test_set_geometry(h.h, kk, tt) == sfar.SFAR_OK
    protos = [args.proto] + ([] if args.only else [p for p in PROTOS if p != args.proto])
    per_proto = {}
    headline = None
    for proto in protos:
        warm_in = [x_dev[0, r] for r in range(w.R)]
        warm_out = [out_dev[0, r] for r in range(w.R)]
        h.allreduce(warm_in, warm_out, proto)
        torch.cuda.synchronize()
        graphs = capture_token_graphs(h, x_dev, out_dev, proto, tokens)
        out_dev.view(torch.int16).fill_(-1)             # every checked output must be written by the replays
        sampler = ClockSampler() if proto == args.proto else None
        ms, clocks = time_graphs(graphs, args.steps, args.warmup, world, sampler)
        check_status(h, proto)
        us = ms * 1000.0 / (args.steps * CALLS_PER_STEP)
        bad = device_mismatches(out_dev, replay_ids, exp_dev[replay_rows])
        per_proto[proto] = {"us_per_call": round(us, 3), "bit_exact": bad == 0, "calls_checked": len(replay_ids),
                            "calls_differing": bad}
        if proto == args.proto:
            headline = (ms, us, clocks, graphs)
        else:
            del graphs
    ms, us, clocks, graphs = headline

    # end to end: host buffers in, result back, through the public API.  Every
    # step copies its own inputs from pinned host memory and its result back;
    # the copies run on their own streams, so step i + 1's inputs arrive while
    # step i computes and step i's result leaves while step i + 1 computes
    # (events order copy-in -> graph -> copy-out of a step, and the reuse of a
    # token's buffers `tokens` steps later)
    stream = torch.cuda.current_stream()
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    out_dev.view(torch.int16).fill_(-1)
    out_host.view(torch.int16).fill_(-1)
    # warm-up: one untimed pass over the steps of the timed loop (the first
    # host-to-device copies of a process ran at a tenth of the later rate)
    for i in range(max(e2e_steps, min(args.warmup, 3)) if e2e_steps else 0):
        t = i % tokens
        sl = slice(t * CALLS_PER_STEP, (t + 1) * CALLS_PER_STEP)
        x_dev[sl].copy_(x_host[sl], non_blocking=True)
        graphs[t].replay()
        out_host[sl].copy_(out_dev[sl], non_blocking=True)
    torch.cuda.synchronize()
    out_host.view(torch.int16).fill_(-1)
    barrier(world)
    s_ev, e_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev_in = [torch.cuda.Event() for _ in range(e2e_steps)]
    ev_done = [torch.cuda.Event() for _ in range(e2e_steps)]
    ev_out = [torch.cuda.Event() for _ in range(e2e_steps)]
    s_ev.record(h2d)
    stream.wait_event(s_ev)
    d2h.wait_event(s_ev)
    for i in range(e2e_steps):
        t = i % tokens
        sl = slice(t * CALLS_PER_STEP, (t + 1) * CALLS_PER_STEP)
        with torch.cuda.stream(h2d):
            if i >= tokens:
                h2d.wait_event(ev_done[i - tokens])        # the graph that last read this token's inputs
            x_dev[sl].copy_(x_host[sl], non_blocking=True)
            ev_in[i].record(h2d)
        stream.wait_event(ev_in[i])
        if i >= tokens:
            stream.wait_event(ev_out[i - tokens])          # the copy that last read this token's outputs
        graphs[t].replay()
        ev_done[i].record(stream)
        with torch.cuda.stream(d2h):
            d2h.wait_event(ev_done[i])
            out_host[sl].copy_(out_dev[sl], non_blocking=True)
            ev_out[i].record(d2h)
    stream.wait_event(ev_out[e2e_steps - 1] if e2e_steps else s_ev)
    d2h.wait_event(ev_done[e2e_steps - 1] if e2e_steps else s_ev)
    e_ev.record(d2h)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(s_ev.elapsed_time(e_ev), world)
    e2e_us = e2e_ms * 1000.0 / (e2e_steps * CALLS_PER_STEP) if e2e_steps else None
    step_bytes = CALLS_PER_STEP * w.R * w.bytes_per_rank
    # the results that reached the host, every rank of every call, against the oracle
    e2e_bad = 0
    for t in e2e_tokens:
        got = inputs.to_bits(out_host[t * CALLS_PER_STEP:(t + 1) * CALLS_PER_STEP])          # [160, R, n]
        want = exp_rows[pos[t] * CALLS_PER_STEP:(pos[t] + 1) * CALLS_PER_STEP]                 # [160, n]
        e2e_bad += int((~(got == want[:, None, :]).all(axis=(1, 2))).sum())
    e2e_ok = e2e_bad == 0 and bool(e2e_tokens)
    del graphs
    k, threads = h.launch(w.n, args.proto)
    h.close()
    del x_dev, out_dev, exp_dev

    floor = floor_probe() if not args.no_floor else {"floor_us": float("nan")}
    large = large_message_roofline(hbm_peak) if not args.no_large else None
    others = other_configs() if not args.no_configs and world == 1 else None

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        from oracle.build import build_oracle
        build_oracle()
        cpu_us, cpu_calls, cpu_s = oracle_cpu_time(x_host, budget_s=args.cpu_seconds)
        cpu = {"value": round(cpu_us, 3), "unit": "us/call", "cores": 1, "kind": "oracle",
               "sample": f"{cpu_calls} calls of R=8 x 8192 bf16 (tp-decode), {cpu_s:.1f} s, single thread"}
        # the same with every host thread splitting each call (a call is short at
        # 16 KB per rank, so thread start-up takes much of what the split saves)
        nthr = os.cpu_count() or 1
        if nthr > 1:
            mt_us, mt_calls, mt_s = oracle_cpu_time(x_host, budget_s=min(3.0, args.cpu_seconds), threads=nthr)
            cpu["threaded"] = {"value": round(mt_us, 3), "unit": "us/call", "cores": nthr,
                               "sample": f"{mt_calls} calls, {mt_s:.1f} s, each split over {nthr} threads"}

    if rank != 0:
        return
    head_ok = per_proto[args.proto]["bit_exact"] and (e2e_ok or not e2e_steps)
    algo_bytes = 2 * w.R * w.bytes_per_rank
    hbm_gbs = algo_bytes / (us * 1e-6) / 1e9
    roofline = {"bound": "latency", "kernel": f"k_{args.proto}", "achieved": round(us, 3),
                "peak": round(floor["floor_us"], 3), "unit": "us/call",
                "frac": round(floor["floor_us"] / us, 4),
                "traffic": profiled_traffic(f"k_{args.proto}"),
                "algorithmic_bytes": algo_bytes, "hbm_achieved_gbs": round(hbm_gbs, 1),
                "hbm_frac": round(hbm_gbs / hbm_peak, 5), "peak_kind": "measured floor (" + peak_kind + " HBM)"}
    line = {"metric": METRIC, "value": round(us, 3) if head_ok else None, "unit": "us/call", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 4),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": workload_config(args, tokens),
            "launch": {"proto": args.proto, "mode": args.mode, "graph": "one CUDA graph per token (160 calls)",
                       "ctas_per_rank": k, "threads_per_cta": threads},
            "bit_exact": head_ok,
            "parity": {"what": "every rank of every call that the warm-up and timed replays computed (and every "
                               "call copied back by the end-to-end loop), compared bit for bit with the oracle",
                       "tokens_replayed": len(replay), "oracle_seconds": round(oracle_check_s, 2)},
            "protocols": per_proto,
            "floor": {k2: (round(v, 3) if isinstance(v, float) else v) for k2, v in floor.items()},
            "vs_floor": round(us / floor["floor_us"], 3),
            "vs_floor_median_pair": (round(us / (floor["empty_kernel_us"] + floor["flag_rtt_median_us"]), 3)
                                     if "flag_rtt_median_us" in floor else None),
            "roofline": roofline, "roofline_large": large, "configs": others,
            "e2e": ({"value": round(e2e_us, 3), "unit": "us/call", "h2d_bytes_per_step": step_bytes,
                     "d2h_bytes_per_step": step_bytes, "steps": e2e_steps, "bit_exact": e2e_ok,
                     "calls_checked": len(e2e_tokens) * CALLS_PER_STEP,
                     "copies": "own streams, overlapping the neighbouring steps' graphs"}
                    if e2e_steps else None),
            "gpu_launches": args.steps * CALLS_PER_STEP,
            "clocks": clocks, "cpu_baseline": cpu}
    print(json.dumps(line), flush=True)
    if not head_ok:
        print(f"bench: {args.proto} results differ from the oracle", file=sys.stderr)
        sys.exit(1)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=640)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--proto", choices=ALL, default="ll", help="headline protocol (the others of the one-shot "
                    "set are timed beside it unless --only)")
    ap.add_argument("--mode", choices=["serial", "overlap", "plain", "cooperative"], default="serial",
                    help="launch mode of the handle (serial: the handle's default)")
    ap.add_argument("--no-large", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--tokens", type=int, default=TOKENS, help="token graphs (inputs cycle over them)")
    ap.add_argument("--only", action="store_true", help="time the headline protocol only")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-floor", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the small and batched-decode workloads")
    ap.add_argument("--geometry", default="", help="CTAS,THREADS override of the launch geometry")
    ap.add_argument("--large-only", action="store_true", help="only the large-message HBM roofline")
    ap.add_argument("--large-r", type=int, default=8)
    ap.add_argument("--large-mb", type=int, default=64)
    ap.add_argument("--large-dtype", choices=["bf16", "fp32"], default="bf16")
    ap.add_argument("--suite-r", type=int, default=0, help="atomic and fused suites: only this rank count")
    ap.add_argument("--suite-rows", type=int, default=0, help="fused suite: only this row count")
    ap.add_argument("--suite-bytes", type=int, default=0, help="latency and atomic suites: only this message size "
                    "per rank")
    ap.add_argument("--suite-protos", default="", help="latency suite: comma list of protocols (default: all)")
    ap.add_argument("--decode-layers", type=int, default=80, help="decode suite: layers per token")
    ap.add_argument("--suite", default="", help="comma list of latency,bandwidth,barriers,atomic,fused,decode: sweeps as JSON lines")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    world, rank, _ = dist_setup(args.gpus)
    if args.suite:
        run_suite(args)
    elif args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

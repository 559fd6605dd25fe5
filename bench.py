"""Benchmark: achieved HBM GB/s and us per fused verify pass.

One step = one fused, ordered verify pass (all products of the layer stack
for N = 8 columns) over the full synthetic workload: 64 layers x (NVFP4
q, k, v, o 5120x5120; NVFP4 gate+up 34816x5120; row-scaled FP8 down
5120x17408) + NVFP4 head 151936x5120 = 16.34 GB of weight+scale bytes read
per pass.  ``value`` is those bytes per second, with weights and x resident
in HBM; ``e2e`` is the same metric through the public API with x copied from
pinned host memory and y copied back inside the timed region.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
For N > 1 it runs under torchrun, one independent replica per GPU (the
product has no exchange step), and rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "achieved HBM GB/s (% of GB300 peak) and µs per NVFP4 verify pass, N=1–8"
WORKLOAD = ("verify stack: 64 layers x (NVFP4 q,k,v,o 5120x5120; NVFP4 gate+up 34816x5120 "
            "as two 17408x5120 halves; row-scaled FP8 down 5120x17408) + NVFP4 head "
            "151936x5120; W ~ N(0,0.02) RTN-quantised, x BF16 ~ N(0,1); seed 4")
FALLBACK_HBM_GBS = 6800.0
WEIGHTS = "nvfp4 / row-scaled fp8-e4m3, decoded exactly to bf16; fp32 accumulation"


def workload_name(args) -> str:
    if args.attn_fmt == "fp8":
        return WORKLOAD.replace("NVFP4 q,k,v,o 5120x5120", "row-scaled FP8 q,k,v,o 5120x5120")
    return WORKLOAD


def stack_bytes(mats) -> int:
    """Algorithmic weight+scale bytes of one pass over `mats` (NVFP4: M*K/2
    codes + M*K/16 scales + 4; row-scaled FP8: M*K codes + 4*M)."""
    return sum(m.M * m.K // 2 + m.M * m.K // 16 + 4 if m.fmt == "nvfp4" else m.M * m.K + 4 * m.M
               for m in mats)


def stack_config(args, world: int) -> dict:
    """The `config` of the JSON line, identical for both arms."""
    from verify_gemm_gb300.inputs import stack_mats

    mats = stack_mats(args.layers, args.attn_fmt)
    return {"workload": workload_name(args), "N": args.N, "mode": "ordered",
            "bytes_per_pass": stack_bytes(mats), "matrices": len(mats),
            "l2": "inputs 16.3 GB per pass >> 129 MB L2; no flush needed",
            "parallelism": f"replicas x{world}"}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    # 200 ordered passes take about 0.85 s: long enough for several clock samples
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--N", type=int, default=8)
    ap.add_argument("--widths", default="1,2,4", help="extra widths reported per pass")
    ap.add_argument("--layers", type=int, default=64)
    ap.add_argument("--attn-fmt", choices=["nvfp4", "fp8"], default="nvfp4",
                    help="stack q,k,v,o format: nvfp4 (16.34 GB pass, the headline) or fp8 "
                         "(row-scaled, the pages' checkpoint mix: 19.28 GB)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the single-product configurations (per_config)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--workload", default="stack",
                    choices=["stack", "fused", "tiny", "proj", "gateup", "down", "head", "probe"],
                    help="stack: the verify pass (headline); fused: the verify pass with RMS "
                         "norms, the gated activation and dependent x; others: one product of "
                         "that configuration, timed alone with an L2 flush between launches")
    ap.add_argument("--fmt", choices=["nvfp4", "fp8", "mxfp8", "int4g"], default=None,
                    help="single products: pack the configuration's weights in this format "
                         "instead of its own")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def profiled_traffic():
    """Per-launch DRAM bytes of the verify kernel from the committed ncu summary."""
    p = os.path.join(ROOT, "profiles", "traffic.txt")
    try:
        with open(p) as f:
            for line in f:
                parts = line.split()
                if len(parts) >= 3 and parts[0] == "stream_kernel" and parts[1] == "verify_stack_N8":
                    return float(parts[2])
    except OSError:
        pass
    return None


class ClockSampler:
    """nvidia-smi clock / throttle samples during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index, interval_ms=20):
        self.gpu = gpu_index
        self.interval = interval_ms
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", str(self.interval)],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                c = [x.strip() for x in line.split(",")]
                if len(c) >= 9:
                    rows.append(c)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": float(rows[0][2]) if rows[0][2].replace(".", "").isdigit() else None,
                "reasons": reasons, "samples": len(rows)}


def dist_init(args):
    from verify_gemm_gb300 import replicas

    ranks = replicas.from_env()
    replicas.init(ranks, "nccl" if args.impl == "ours" else "gloo")
    return ranks.world, ranks.rank, ranks.local


def pcts(xs, qs):
    """Nearest-rank percentiles of xs for each q in qs (0..100)."""
    v = sorted(xs)
    return [v[min(len(v) - 1, max(0, int(round(q / 100 * (len(v) - 1)))))] for q in qs]


def barrier(world):
    from verify_gemm_gb300 import replicas

    replicas.barrier(replicas.Ranks(world=world))


def max_over_ranks(v, world, device=None):
    from verify_gemm_gb300 import replicas

    return replicas.max_over_ranks(v, replicas.Ranks(world=world), device)


# ------------------------------------------------------------- CPU oracle

_CPU_SAMPLE = None


def _cpu_sample_inputs():
    """The oracle's inputs for cpu_sample, drawn and quantised once."""
    global _CPU_SAMPLE
    if _CPU_SAMPLE is None:
        import numpy as np
        import torch

        import oracle
        from verify_gemm_gb300.inputs import HIDDEN, INTERMEDIATE, generator, draw_weight, draw_x

        orc = oracle.get()
        g = generator(4)
        Wq = draw_weight(g, HIDDEN, HIDDEN).numpy()
        Wd = draw_weight(g, HIDDEN, INTERMEDIATE).numpy()
        Wh = draw_weight(g, 2048, HIDDEN).numpy()
        x5 = draw_x(g, 8, HIDDEN).view(torch.int16).numpy().view(np.uint16)
        x17 = draw_x(g, 8, INTERMEDIATE).view(torch.int16).numpy().view(np.uint16)
        nbytes = SAMPLE_BYTES
        _CPU_SAMPLE = (orc, orc.nvfp4_quantise(Wq), orc.fp8_quantise(Wd), orc.nvfp4_quantise(Wh),
                       x5, x17, nbytes)
    return _CPU_SAMPLE


# 14,745,604 + 89,149,440 + 5,898,240 weight+scale bytes
SAMPLE_BYTES = (5120 * 5120 * 9 // 16 + 4) + (5120 * 17408 + 4 * 5120) + 2048 * 5120 * 9 // 16
SAMPLE_TEXT = ("oracle FP64 GEMV, N=8, on layer-0 q (NVFP4 5120x5120), down (FP8 5120x17408) "
               f"and 2048 head rows (NVFP4 2048x5120): {SAMPLE_BYTES:,} weight+scale bytes "
               "per round")


def cpu_round(threads: int) -> float:
    """One round of the oracle over the bounded sample; returns seconds."""
    orc, (nq, sq, gq), (qd, rd), (nh, sh, gh), x5, x17, _ = _cpu_sample_inputs()
    t0 = time.perf_counter()
    orc.gemv_nvfp4(nq, sq, gq, x5, threads=threads)
    orc.gemv_fp8(qd, rd, x17, threads=threads)
    orc.gemv_nvfp4(nh, sh, gh, x5, threads=threads)
    return time.perf_counter() - t0


def cpu_sample(seconds: float):
    """Time the CPU oracle's GEMV on a bounded sample of the workload: the
    first layer's q (NVFP4 5120x5120) and down (FP8 5120x17408) and 2048 rows
    of the head, N = 8, all host threads, repeated for about `seconds`; then
    one round on a single thread."""
    orc, (nq, sq, gq), (qd, rd), (nh, sh, gh), x5, x17, nbytes = _cpu_sample_inputs()
    threads = os.cpu_count() or 1
    done = 0
    t0 = time.perf_counter()
    while True:
        orc.gemv_nvfp4(nq, sq, gq, x5, threads=threads)
        orc.gemv_fp8(qd, rd, x17, threads=threads)
        orc.gemv_nvfp4(nh, sh, gh, x5, threads=threads)
        done += nbytes
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    one = cpu_round(1)
    return {"value": done / el / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{SAMPLE_TEXT}; {done / nbytes:.0f} rounds in {el:.1f} s on all threads",
            "single_thread": {"value": nbytes / one / 1e9, "unit": "GB/s", "cores": 1,
                              "sample": "one round of the same sample"}}


def run_reference_config(args):
    """The oracle (as it stands) on one single-product configuration in
    full: its weights quantised by the oracle, then GEMV rounds on all host
    threads for at least a second, and one round on one thread."""
    import numpy as np
    import torch

    import oracle
    from verify_gemm_gb300.inputs import WORKLOADS, draw_workload

    orc = oracle.get()
    key = {"down": "down_head", "head": "down_head"}.get(args.workload, args.workload)
    title, names = SINGLE[args.workload]
    Ws, xs = draw_workload(key, args.N)
    jobs, nbytes = [], 0
    for m, W in zip(WORKLOADS[key].mats, Ws):
        if m.name not in names:
            continue
        xb = xs[m.K].view(torch.int16).numpy().view(np.uint16)
        if m.fmt == "nvfp4":
            nib, sc, gs = orc.nvfp4_quantise(W.numpy())
            jobs.append(lambda t, a=(nib, sc, gs, xb): orc.gemv_nvfp4(*a, threads=t))
            nbytes += m.M * m.K // 2 + m.M * m.K // 16 + 4
        else:
            q, rs = orc.fp8_quantise(W.numpy())
            jobs.append(lambda t, a=(q, rs, xb): orc.gemv_fp8(*a, threads=t))
            nbytes += m.M * m.K + 4 * m.M
    del Ws
    threads = os.cpu_count() or 1

    def one(t):
        t0 = time.perf_counter()
        for j in jobs:
            j(t)
        return time.perf_counter() - t0

    one(threads)
    per = []
    while sum(per) < 1.0:
        per.append(one(threads))
    single = one(1)
    med = statistics.median(per)
    print(json.dumps({"impl": "reference", "metric": METRIC, "unit": "GB/s",
                      "config": {"workload": title, "N": args.N, "bytes": nbytes},
                      "value": nbytes / med / 1e9, "ms_per_step": med * 1e3, "cores": threads,
                      "rounds": len(per),
                      "single_thread": {"value": nbytes / single / 1e9, "ms": single * 1e3}}),
          flush=True)


def run_reference(args, world, rank):
    """The reference arm: the CPU oracle as it stands, on all host threads.
    Each step is one round of the bounded sample (about 0.1 s); the line
    reports what was timed: the sample's GB/s and the measured seconds per
    round.  The time a full 16.34 GB pass would take at that rate is
    reported separately and labelled as extrapolated."""
    if rank != 0:
        return
    threads = os.cpu_count() or 1
    _cpu_sample_inputs()
    nbytes = _cpu_sample_inputs()[-1]
    for _ in range(args.warmup):
        cpu_round(threads)
    per = [cpu_round(threads) for _ in range(args.steps)]
    total = sum(per)
    value = nbytes * args.steps / total / 1e9
    one = cpu_round(1)
    cfg = stack_config(args, world)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": total / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": cfg,
            "step": "one round of the oracle over the bounded sample (timed); "
                    + SAMPLE_TEXT,
            "extrapolated_full_pass_ms": cfg["bytes_per_pass"] / (value * 1e9) * 1e3,
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": f"{SAMPLE_TEXT}; {args.steps} rounds",
                             "single_thread": {"value": nbytes / one / 1e9, "unit": "GB/s",
                                               "cores": 1,
                                               "sample": "one round of the same sample"}},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------- GPU

def run_ours(args, world, rank, local):
    import torch

    import verify_gemm_gb300 as vg
    from verify_gemm_gb300 import build as vbuild
    from verify_gemm_gb300.workloads import build_stack
    from verify_gemm_gb300 import replicas

    vbuild.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    st = build_stack(args.N, device=dev, layers=args.layers, attn_fmt=args.attn_fmt)
    plan = st.plan(ordered=True)
    nbytes = st.bytes
    torch.cuda.synchronize()

    def timed(run, steps, warmup):
        for _ in range(warmup):
            run()
        torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
        evs[0].record(stream)
        for i in range(steps):
            run()
            evs[i + 1].record(stream)
        torch.cuda.synchronize()
        barrier(world)
        per = [evs[i].elapsed_time(evs[i + 1]) for i in range(steps)]
        return sum(per), per

    clocks = ClockSampler(local)
    clocks.start()
    total_ms, per = timed(plan.run, args.steps, args.warmup)
    clk = clocks.stop()
    if plan.check() != 0:
        raise RuntimeError("verify pass reported a device error")
    # the same passes back to back for at least one second, with their own
    # clock record: a steadier view of the clocks than a short timed region
    reps = max(args.steps, int(1.0 / max(1e-4, total_ms / args.steps / 1e3)) + 1)
    clocks2 = ClockSampler(local)
    clocks2.start()
    s_ms, _ = timed(plan.run, reps, 0)
    clk2 = clocks2.stop()
    if plan.check() != 0:
        raise RuntimeError("verify pass reported a device error")
    sustained = {"passes": reps, "ms": round(s_ms, 1),
                 "GBps": round(nbytes * reps / (s_ms / 1e3) / 1e9, 1), "clocks": clk2}
    total_ms = max_over_ranks(total_ms, world, dev)
    value = replicas.job_gbps(nbytes, args.steps, total_ms, replicas.Ranks(world=world))
    kernel_ms = statistics.mean(per)
    achieved = nbytes / (kernel_ms / 1e3) / 1e9
    peak, peak_kind = peaks()

    extra = {}
    unordered = st.plan(ordered=False)
    u_ms, _ = timed(unordered.run, max(3, args.steps // 2), 2)
    unordered.close()
    extra["unordered_gbs"] = nbytes * max(3, args.steps // 2) / (u_ms / 1e3) / 1e9
    # the other widths through the same plan: each pass reads its width from
    # a device word (no new plan, no host-side width)
    widths = {}
    width = torch.zeros(1, dtype=torch.int32, device=dev)
    plan.set_width(width)
    for w in [int(v) for v in args.widths.split(",") if v]:
        if w == args.N or w > args.N:
            continue
        width.fill_(w)
        ms, _ = timed(plan.run, max(3, args.steps // 2), 2)
        if plan.check() != 0:
            raise RuntimeError("verify pass reported a device error")
        us = ms / max(3, args.steps // 2) * 1e3
        widths[str(w)] = {"us_per_pass": round(us, 1), "GBps": round(nbytes / us / 1e3, 1)}
    plan.set_width(None)
    widths[str(args.N)] = {"us_per_pass": round(total_ms / args.steps * 1e3, 1),
                           "GBps": round(nbytes / (total_ms / args.steps) / 1e6, 1)}

    # one draft step (row-scaled FP8 layer + NVFP4 head) at N = 1
    draft = None
    if not args.no_configs:
        from verify_gemm_gb300.inputs import DRAFT_SEED, draft_mats

        ds = build_stack(1, device=dev, mats=draft_mats(), seed=DRAFT_SEED)
        dplan = ds.plan(ordered=True)
        ms, per_d = timed(dplan.run, args.steps, args.warmup)
        if dplan.check() != 0:
            raise RuntimeError("draft step reported a device error")
        dplan.close()
        med = statistics.median(per_d)
        draft = {"workload": "draft step: row-scaled FP8 q,k,v,o 5120x5120, gate+up "
                             "2x17408x5120, down 5120x17408 + NVFP4 head 151936x5120, N=1, "
                             "ordered; seed 5",
                 "bytes": ds.bytes, "us_per_step": round(1e3 * med, 1),
                 "us_p10_p90": [round(1e3 * q, 1) for q in pcts(per_d, (10, 90))],
                 "GBps": round(ds.bytes / (med / 1e3) / 1e9, 1)}
        del ds
        torch.cuda.empty_cache()

    # the same stack verified 16 columns wide (e.g. four requests' rounds of
    # one token and three drafts) in one pass
    wide = None
    if not args.no_configs and args.layers == 64 and args.N <= 8:
        wst = build_stack(16, device=dev, attn_fmt=args.attn_fmt)
        wpl = wst.plan(ordered=True)
        ms, per_w = timed(wpl.run, args.steps, args.warmup)
        if wpl.check() != 0:
            raise RuntimeError("wide stack reported a device error")
        wpl.close()
        med = statistics.median(per_w)
        wide = {"N": 16, "bytes": wst.bytes, "us_per_pass": round(1e3 * med, 1),
                "GBps": round(wst.bytes / (med / 1e3) / 1e9, 1)}
        del wst
        torch.cuda.empty_cache()

    # the same stack with every matrix in MXFP8, then in groupwise INT4
    format_stacks = None
    if not args.no_configs and args.layers == 64:
        format_stacks = {}
        for f in ("mxfp8", "int4g"):
            fst = build_stack(args.N, device=dev, all_fmt=f)
            fpl = fst.plan(ordered=True)
            ms, per_s = timed(fpl.run, args.steps, args.warmup)
            if fpl.check() != 0:
                raise RuntimeError("format stack reported a device error")
            fpl.close()
            med = statistics.median(per_s)
            format_stacks[f] = {"bytes": fst.bytes, "us_per_pass": round(1e3 * med, 1),
                                "GBps": round(fst.bytes / (med / 1e3) / 1e9, 1)}
            del fst
            torch.cuda.empty_cache()

    # the same stack with its neighbours fused in and real dependencies:
    # RMS norm -> q,k,v (x = the norm's y); o; RMS norm -> gate+up with the
    # gated activation -> down (x = the activation's y); final norm -> head
    fused = None
    if not args.no_configs and args.layers == 64:
        from verify_gemm_gb300.workloads import build_fused_stack

        fs = build_fused_stack(args.N, device=dev, attn_fmt=args.attn_fmt)
        fplan = fs.plan()
        ms, per_f = timed(fplan.run, args.steps, args.warmup)
        if fplan.check() != 0:
            raise RuntimeError("fused stack reported a device error")
        fplan.close()
        med = statistics.median(per_f)
        fused = {"workload": "the verify stack with RMS norms before q,k,v and before the MLP, "
                             "the gated activation fused into gate+up and written as down's x, "
                             "a final norm before the head; every dependent x copied only after "
                             "its producer group completes",
                 "N": args.N, "bytes": fs.bytes, "phases": len({e.group for e in fs.entries}),
                 "us_per_pass": round(1e3 * med, 1),
                 "us_p10_p90": [round(1e3 * q, 1) for q in pcts(per_f, (10, 90))],
                 "GBps": round(fs.bytes / (med / 1e3) / 1e9, 1)}
        del fs
        torch.cuda.empty_cache()

    e2e = None
    if not args.no_e2e:
        x_host = torch.empty(st.x_all.shape, dtype=st.x_all.dtype, pin_memory=True)
        x_host.copy_(st.x_all)
        y_host = torch.empty(st.y_all.shape, dtype=st.y_all.dtype, pin_memory=True)

        # Each step uploads its x from pinned host memory, runs the pass and
        # reads its y back.  Two buffer pairs (and two plans) alternate, so
        # step i's upload overlaps pass i-1 and its read-back overlaps pass
        # i+1, on their own streams; every byte still moves inside the timed
        # region, which ends when the last read-back has landed.
        st2 = st.with_new_buffers()
        sets = [(st, plan), (st2, st2.plan(ordered=True))]
        y_hosts = [y_host, torch.empty_like(y_host, pin_memory=True)]
        up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_x = [torch.cuda.Event() for _ in range(2)]
        ev_pass = [torch.cuda.Event() for _ in range(2)]
        ev_y = [torch.cuda.Event() for _ in range(2)]

        def e2e_steps(n):
            for i in range(n):
                k = i % 2
                cur, cur_plan = sets[k]
                up.wait_event(ev_pass[k])        # pass i-2 used this pair
                with torch.cuda.stream(up):
                    cur.x_all.copy_(x_host, non_blocking=True)
                    ev_x[k].record(up)
                stream.wait_event(ev_x[k])
                stream.wait_event(ev_y[k])       # y of pass i-2 has been read back
                cur_plan.run()
                ev_pass[k].record(stream)
                down.wait_event(ev_pass[k])
                with torch.cuda.stream(down):
                    y_hosts[k].copy_(cur.y_all, non_blocking=True)
                    ev_y[k].record(down)
            stream.wait_event(ev_y[(n - 1) % 2])
            stream.wait_event(ev_y[n % 2])

        e2e_steps(args.warmup)
        torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        up.wait_event(e0)
        down.wait_event(e0)
        e2e_steps(args.steps)
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        e_ms = e0.elapsed_time(e1)
        # both pairs hold the same x, so the y read back must match bit for bit
        e2e_y_match = bool(torch.equal(y_hosts[0], y_hosts[1]))
        for _, p2 in sets[1:]:
            p2.close()
        e_ms = max_over_ranks(e_ms, world, dev)
        e2e = {"value": replicas.job_gbps(nbytes, args.steps, e_ms, replicas.Ranks(world=world)),
               "unit": "GB/s",
               "h2d_bytes_per_step": st.x_all.numel() * 2,
               "d2h_bytes_per_step": st.y_all.numel() * 2,
               "overlapped": "two buffer pairs; uploads and read-backs on their own streams",
               "y_read_back_consistent": e2e_y_match}
    plan.close()

    configs = per_config(20, 3) if (rank == 0 and not args.no_configs) else None
    cb = None
    if rank == 0 and world == 1:
        cb = cpu_sample(args.cpu_seconds)
    if rank == 0:
        cfg = stack_config(args, world)
        assert cfg["bytes_per_pass"] == nbytes, (cfg["bytes_per_pass"], nbytes)
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(total_ms / args.steps, 4),
            # this rank's per-pass times (events between passes), p10 / p50 / p90
            "us_per_step_p10_p50_p90": [round(1e3 * q, 1) for q in pcts(per, (10, 50, 90))],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "weights": WEIGHTS, "data": "synthetic",
            "config": cfg,
            "pct_of_8TBps": round(100 * value / world / 8000, 1),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                         "unit": "GB/s", "frac": round(achieved / peak, 4),
                         "traffic": (profiled_traffic() if (args.attn_fmt, args.N, args.layers)
                                     == ("nvfp4", 8, 64) else None),
                         "peak_kind": peak_kind + " (MEASURED_PEAKS hbm_gbs, copy)"},
            "per_width": widths, **extra,
            "per_config": configs, "draft_step": draft, "fused_stack": fused,
            "format_stacks": format_stacks, "wide_stack": wide,
            "sustained": sustained,
            "e2e": e2e, "gpu_launches": args.steps, "clocks": clk,
        }
        if cb is not None:
            line["cpu_baseline"] = cb
        print(json.dumps(line), flush=True)


SINGLE = {
    "tiny": ("tiny NVFP4 GEMV 256x512, seed 0", ["w"]),
    "proj": ("single projection NVFP4 5120x5120, outlier x, seed 1", ["w"]),
    "gateup": ("fused gate+up NVFP4 34816x5120 (two 17408x5120 halves), seed 2",
               ["gate", "up"]),
    "down": ("row-scaled FP8 down 5120x17408, seed 3", ["down"]),
    "head": ("NVFP4 head 151936x5120, seed 3", ["head"]),
}
# the single-product configurations and the widths each is quoted at; the
# last entries time the same shapes in the other weight formats
PER_CONFIG = [("tiny", (1,)), ("proj", (1,)), ("gateup", (1, 2, 4, 8, 16, 32)),
              ("down", (1, 8, 16)), ("head", (1, 8, 16, 32)), ("proj", (8,), "mxfp8"),
              ("proj", (8,), "int4g"),
              ("gateup", (8,), "mxfp8"), ("gateup", (8,), "int4g"), ("head", (8,), "mxfp8"),
              ("head", (8,), "int4g")]


def time_single(workload: str, N: int, steps: int, warmup: int, flush, fmt=None):
    """One configuration's product, timed alone: L2 flushed (a 512 MB write)
    before every launch, CUDA events around each launch only; fmt: the
    weights in that format instead of the configuration's.  Returns (bytes,
    per-launch ms list)."""
    import torch

    import verify_gemm_gb300 as vg
    from verify_gemm_gb300.inputs import WORKLOADS, draw_workload

    key = {"down": "down_head", "head": "down_head"}.get(workload, workload)
    _, names = SINGLE[workload]
    Ws, xs = draw_workload(key, N, device="cuda")
    entries = []
    for m, W in zip(WORKLOADS[key].mats, Ws):
        if m.name not in names:
            continue
        from verify_gemm_gb300.workloads import pack

        wt = pack(W, fmt or m.fmt)
        y = torch.empty((N, m.M), dtype=torch.bfloat16, device="cuda")
        entries.append((wt, xs[m.K], y, 0))
    del Ws
    nbytes = sum(e[0].nbytes for e in entries)
    plan = None
    if len(entries) == 1:
        wt, x, y, _ = entries[0]
        ws = vg.workspace_for(wt, N=N)

        def run():
            vg.gemv(wt, x, y, ws)
    else:
        plan = vg.VerifyPlan(entries, N, ordered=True)
        run = plan.run
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        flush.fill_(1)
        run()
    torch.cuda.synchronize()
    per = []
    for i in range(steps):
        flush.fill_(i & 0xFF)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        run()
        b.record(stream)
        per.append((a, b))
    torch.cuda.synchronize()
    ms = [a.elapsed_time(b) for a, b in per]
    if plan is not None:
        if plan.check() != 0:
            raise RuntimeError("verify pass reported a device error")
        plan.close()
    elif vg.workspace_error(ws) != 0:
        raise RuntimeError("GEMV reported a device error")
    return nbytes, ms


def run_single(args, local):
    """One configuration's product, timed alone with an L2 flush between
    launches (a 512 MB write)."""
    import torch

    from verify_gemm_gb300 import build as vbuild

    vbuild.build()
    torch.cuda.set_device(local)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    nbytes, ms = time_single(args.workload, args.N, args.steps, args.warmup, flush, fmt=args.fmt)
    med = statistics.median(ms)
    peak, kind = peaks()
    title, _ = SINGLE[args.workload]
    if args.fmt:
        title = f"{title}, weights packed as {args.fmt}"
    line = {"metric": METRIC, "value": round(nbytes / (med / 1e3) / 1e9, 1), "unit": "GB/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(med, 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "weights": WEIGHTS,
            "data": "synthetic",
            "config": {"workload": title, "N": args.N, "bytes": nbytes, "fmt": args.fmt,
                       "l2": "flushed by a 512 MB write before every launch",
                       "us_p10_p90": [round(1e3 * q, 2) for q in pcts(ms, (10, 90))]},
            "roofline": {"bound": "hbm", "achieved": round(nbytes / (med / 1e3) / 1e9, 1),
                         "peak": peak, "unit": "GB/s",
                         "frac": round(nbytes / (med / 1e3) / 1e9 / peak, 4), "traffic": None,
                         "peak_kind": kind},
            "gpu_launches": args.steps}
    print(json.dumps(line), flush=True)


def run_fused(args, local):
    """The fused verify stack alone (RMS norms, the gated activation, dependent
    x; --layers layers, --N columns), ordered, one pass per step.  With 64
    layers its 16.3 GB exceed L2; a smaller stack is for profiling."""
    import torch

    from verify_gemm_gb300 import build as vbuild
    from verify_gemm_gb300.workloads import build_fused_stack

    vbuild.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    fs = build_fused_stack(args.N, layers=args.layers, device=dev, attn_fmt=args.attn_fmt)
    plan = fs.plan()
    for _ in range(args.warmup):
        plan.run()
    torch.cuda.synchronize()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    evs[0].record(stream)
    for i in range(args.steps):
        plan.run()
        evs[i + 1].record(stream)
    torch.cuda.synchronize()
    if plan.check() != 0:
        raise RuntimeError("fused stack reported a device error")
    plan.close()
    ms = [evs[i].elapsed_time(evs[i + 1]) for i in range(args.steps)]
    med = statistics.median(ms)
    peak, kind = peaks()
    gbps = fs.bytes / (med / 1e3) / 1e9
    line = {"metric": METRIC, "value": round(gbps, 1), "unit": "GB/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(med, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "weights": WEIGHTS, "data": "synthetic",
            "config": {"workload": f"fused verify stack, {args.layers} layers: RMS norms, "
                                   "gated activation, dependent x",
                       "N": args.N, "bytes": fs.bytes,
                       "phases": len({e.group for e in fs.entries}),
                       "us_p10_p90": [round(1e3 * q, 1) for q in pcts(ms, (10, 90))]},
            "roofline": {"bound": "hbm", "achieved": round(gbps, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(gbps / peak, 4), "traffic": None, "peak_kind": kind},
            "gpu_launches": args.steps}
    print(json.dumps(line), flush=True)


def per_config(steps: int, warmup: int):
    """Every single-product configuration at every width it is quoted at,
    timed alone (median of `steps` launches, L2 flushed before each)."""
    import torch

    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    out = {}
    for wl, widths, *fmt in PER_CONFIG:
        for N in widths:
            nbytes, ms = time_single(wl, N, steps, warmup, flush, *fmt)
            med = statistics.median(ms)
            out[f"{wl}{' ' + fmt[0] if fmt else ''} N={N}"] = {"us": round(1e3 * med, 2),
                                  "us_p10_p90": [round(1e3 * q, 2) for q in pcts(ms, (10, 90))],
                                  "GBps": round(nbytes / (med / 1e3) / 1e9, 1), "bytes": nbytes}
            torch.cuda.empty_cache()
    del flush
    return out


def run_probe(args, local):
    """Read-only HBM ceiling: vector loads and per-warp bulk-copy rings over a
    4 GiB buffer (>> L2), median of `steps` launches each."""
    import ctypes

    import torch

    from verify_gemm_gb300 import _lib
    from verify_gemm_gb300 import build as vbuild

    vbuild.build()
    torch.cuda.set_device(local)
    lib = _lib.load()
    nbytes = 4 << 30
    buf = torch.ones(nbytes // 4, dtype=torch.int32, device="cuda")
    sink = torch.zeros(8192, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    out = {}
    configs = [(1, 12288, 1), (0, 0, 0), (1, 4096, 2), (2, 4096, 3), (2, 4096, 2),
               (2, 8192, 1), (3, 4096, 2), (3, 2048, 4), (3, 8192, 1), (2, 12288, 1)]
    for mode, chunk, slots in configs:
        ms = []
        for i in range(args.warmup + args.steps):
            a, b = torch.cuda.Event(True), torch.cuda.Event(True)
            a.record(stream)
            s = lib.vg_hbm_read_probe(ctypes.c_void_p(buf.data_ptr()), nbytes, mode, chunk, slots,
                                      ctypes.c_void_p(sink.data_ptr()), sink.numel(),
                                      ctypes.c_void_p(stream.cuda_stream))
            _lib.check(s, "vg_hbm_read_probe")
            b.record(stream)
            torch.cuda.synchronize()
            if i >= args.warmup:
                ms.append(a.elapsed_time(b))
        key = "ldg128" if mode == 0 else \
            f"bulk {chunk}B x{slots} slots/warp, " + \
            {1: "interleaved", 2: "per-block ranges", 3: "per-block ranges + 1/8 side copy"}[mode]
        out.setdefault(key, []).append(round(nbytes / (statistics.median(ms) / 1e3) / 1e9, 1))
    peak, kind = peaks()
    print(json.dumps({"metric": "read-only HBM probe GB/s", "unit": "GB/s", "bytes": nbytes,
                      "results": out, "copy_peak": peak, "peak_kind": kind}), flush=True)


def main():
    args = parse()
    if args.workload == "probe":
        run_probe(args, int(os.environ.get("LOCAL_RANK", "0")))
        return
    world, rank, local = dist_init(args)
    if args.impl == "reference" and args.workload == "fused":
        if rank == 0:
            print(json.dumps({"impl": "reference", "unavailable": "the oracle's fused chain is "
                              "checked in the tests, not timed"}), flush=True)
    elif args.impl == "reference" and args.workload != "stack" and args.fmt:
        if rank == 0:
            print(json.dumps({"impl": "reference", "unavailable": "the oracle's timing runs each "
                              "configuration in its own format"}), flush=True)
    elif args.impl == "reference" and args.workload != "stack":
        if rank == 0:
            run_reference_config(args)
    elif args.impl == "reference":
        run_reference(args, world, rank)
    elif args.workload == "fused":
        run_fused(args, local)
    elif args.workload != "stack":
        run_single(args, local)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()

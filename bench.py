"""Benchmark of the DSpark draft-sample -> schedule -> verify hot path.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                [--workload dspark5]

One step = one decoding round for the whole batch: draft sampling of all G
positions, calibration + prefix scheduling, and verification, on inputs
already resident in HBM.  `value` is verified draft positions (sum of the
scheduled verify lengths) per second over all ranks; the HBM figure is the
algorithmic bytes of the round over the step time.  The e2e figure is the
same metric with the per-round inputs copied from pinned host memory and the
emitted tokens copied back inside the timed region.  Multi-GPU runs are
independent replicas (one batch per rank, weak scaling, no collective on the
data path); `--impl reference` times the CPU oracle on a bounded sample.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "verified draft positions/sec & achieved HBM GB/s at V=129280, B=256, γ=5"
UNIT = "positions/s"


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "25"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def stop(self, region=None):
        """Summary of the samples; with region = (t0, t1) (time.monotonic of the
        timed region's start and end), of those read inside it."""
        if self.proc is None:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=["nvidia-smi unavailable"], samples=0)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        return summarize_clocks(self.lines, region)


def summarize_clocks(lines, region=None):
    """Median SM clock, maximum clock and active slowdown reasons of nvidia-smi
    csv samples [(host time, line)].  With region = (t0, t1), only the samples
    read inside it (plus one 25 ms sampling period after t1, the reader's lag)
    count when there are any; `samples_in_region` says how many there were."""
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def parse(sel):
        sm, smax, reasons = [], [], set()
        for _, ln in sel:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, p in zip(names, parts[3:7]):
                if p.lower() == "active":
                    reasons.add(n)
        return sm, smax, reasons

    inside = [] if region is None else [x for x in lines if region[0] <= x[0] <= region[1] + 0.025]
    sm, smax, reasons = parse(inside)
    n_in = len(sm)
    if not sm:  # the region was shorter than the sampling period
        sm, smax, reasons = parse(lines)
    return dict(sm_mhz=statistics.median(sm) if sm else None, sm_max_mhz=max(smax) if smax else None,
                reasons=sorted(reasons), samples=len(sm), samples_in_region=n_in)


def _dist_init(n):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def _barrier(world):
    if world > 1:
        import torch.distributed as dist
        if dist.get_backend() == "nccl":
            dist.barrier(device_ids=[torch.cuda.current_device()])
        else:
            dist.barrier()


def _max_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _sum_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# --------------------------------------------------------------------------
# CPU oracle leg (cpu_baseline and --impl reference)
# --------------------------------------------------------------------------

def oracle_sample(w, h, seed, budget_s=12.0, threads=None):
    """Time the oracle on a growing sample of requests of workload ``w``."""
    import oracle
    oracle.build()
    threads = threads or len(os.sched_getaffinity(0))
    t0 = time.perf_counter()
    sch = oracle.schedule(h["conf_logits"], h["pos_temp"], h["sps"], w.L_min, w.G) if w.scheduler else None
    t_sched = time.perf_counter() - t0
    vl_all = sch["verify_len"] if sch is not None else np.full(w.B, w.G, np.int32)
    n = min(w.B, max(threads, 8))
    elapsed, done, positions = 0.0, 0, 0
    rid_all = h["request_id"].numpy().astype(np.uint32)
    if "_f64" not in h:  # the weights in the oracle's input precision, converted once
        h["_f64"] = (oracle._f64(h["e_in"]), oracle._f64(h["w_out"]))
    e_in, w_out = h["_f64"]
    while done < w.B:
        reqs = np.arange(done, min(w.B, done + n))
        t0 = time.perf_counter()
        d = oracle.draft_sample_parallel(h["base"][reqs], e_in, w_out, h["anchor"][reqs],
                                         h["temperature"][reqs], rid_all[reqs], seed, threads=threads)
        oracle.verify_parallel(h["target"][reqs], h["base"][reqs], e_in, w_out, h["anchor"][reqs],
                               d["tokens"], vl_all[reqs], h["temperature"][reqs], rid_all[reqs], seed,
                               threads=threads)
        dt = time.perf_counter() - t0
        elapsed += dt
        done += len(reqs)
        positions += int(vl_all[reqs].sum())
        if elapsed >= budget_s:
            break
        remaining = budget_s - elapsed
        per_req = dt / len(reqs)
        n = int(max(1, min(w.B - done, remaining / max(per_req, 1e-9))))
    total = elapsed + t_sched
    return dict(value=positions / total, unit=UNIT, cores=threads, kind="oracle",
                sample="%d of %d requests of one %s round (draft + verify per request, scheduler on "
                       "all requests), %.1f s" % (done, w.B, w.name, total),
                seconds=total, positions=positions)


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo), or None."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip() == "Model name":
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return None


def cpu_baseline_line(w, h, seed, budget_s):
    """The oracle on all host cores (the reported baseline) and on one core."""
    cb = oracle_sample(w, h, seed, budget_s=budget_s)
    c1 = oracle_sample(w, h, seed, budget_s=max(2.0, budget_s / 3), threads=1)
    return dict(value=cb["value"], unit=UNIT, cores=cb["cores"], kind="oracle", sample=cb["sample"],
                cpu_model=cpu_model(),
                single_thread=dict(value=c1["value"], unit=UNIT, cores=1, sample=c1["sample"]))


def run_reference(args, w):
    if int(os.environ.get("RANK", "0")) != 0:
        return
    from speculative_decoding_draft_head_gb300.synth import make_inputs
    h = make_inputs(w, args.seed, device="cpu")
    vals = []
    info = None
    for i in range(args.warmup + args.steps):
        # about 90 s in all; a step is at least one batch of requests
        budget = max(0.05, 90.0 / max(1, args.warmup + args.steps))
        r = oracle_sample(w, h, args.seed, budget_s=budget)
        if i >= args.warmup:
            vals.append(r["value"])
            info = r
    value = float(np.mean(vals))
    line = dict(impl="reference", metric=METRIC, value=value, unit=UNIT, n_gpus=args.gpus,
                steps=args.steps, warmup=args.warmup, ms_per_step=1000.0 * info["seconds"],
                higher_is_better=True, scaling="weak", vs_baseline=None, dtype="f64", data="synthetic",
                config=_config(w),
                cpu_baseline=dict(value=value, unit=UNIT, cores=info["cores"], kind="oracle",
                                  sample=info["sample"], cpu_model=cpu_model()),
                e2e=dict(value=value, unit=UNIT, h2d_bytes_per_step=0, d2h_bytes_per_step=0))
    print(json.dumps(line))


def _config(w):
    return dict(workload="%s: B=%d, gamma=%d, V=%d, r=%d, %s logits" % (w.name, w.B, w.G, w.V, w.r, w.dtype),
                B=w.B, gamma=w.G, V=w.V, r=w.r, storage=w.dtype, scheduler=w.scheduler,
                l2="inputs larger than L2 (base and target logits > 129 MB); W_out stays L2-resident")


# --------------------------------------------------------------------------
# GPU leg
# --------------------------------------------------------------------------

def run_ours(args, w):
    from speculative_decoding_draft_head_gb300 import binding
    from speculative_decoding_draft_head_gb300.synth import make_inputs

    rank, world, local = _dist_init(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    binding.load()
    inp = make_inputs(w, args.seed + rank, device=dev, request_id_base=rank * w.B)
    stream = torch.cuda.current_stream(dev)
    s_ = 2 if w.dtype == "bf16" else 4
    B, G, V, r = w.B, w.G, w.V, w.r

    ws_d = binding.default_workspace(binding.WS_DRAFT, B, G, V, r, dev)
    ws_s = binding.default_workspace(binding.WS_SCHEDULE, B, G, 8, 1, dev)
    ws_v = binding.default_workspace(binding.WS_VERIFY, B, G, V, r, dev)
    d_out = dict(tokens=torch.empty((B, G), dtype=torch.int32, device=dev),
                 lse=torch.empty((B, G), dtype=torch.float32, device=dev),
                 logq=torch.empty((B, G), dtype=torch.float32, device=dev))
    s_out = dict(conf=torch.empty((B, G), dtype=torch.float32, device=dev),
                 cum_conf=torch.empty((B, G), dtype=torch.float32, device=dev),
                 verify_len=torch.full((B,), G, dtype=torch.int32, device=dev),
                 theta=torch.empty((1,), dtype=torch.float64, device=dev))
    v_out = dict(accept_len=torch.empty((B,), dtype=torch.int32, device=dev),
                 out_tokens=torch.empty((B, G + 1), dtype=torch.int32, device=dev),
                 num_out=torch.empty((B,), dtype=torch.int32, device=dev),
                 target_lse=torch.empty((B, G + 1), dtype=torch.float32, device=dev),
                 logp=torch.empty((B, G), dtype=torch.float32, device=dev))

    ev = {k: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for k in ("draft", "sched", "verify")}
    call_ms = {k: [] for k in ev}

    def step(x, timed=False, st=None):
        st = stream if st is None else st
        if timed:
            ev["draft"][0].record(stream)
        binding.draft_sample(x["base"], x["e_in"], x["w_out"], x["anchor"], x["temperature"],
                             x["request_id"], args.seed, out=d_out, workspace=ws_d, stream=st)
        if timed:
            ev["draft"][1].record(stream)
            ev["sched"][0].record(stream)
        vl = None
        if w.scheduler:
            binding.schedule_prefix(x["conf_logits"], x["pos_temp"], x["sps"], w.L_min, G, out=s_out,
                                    workspace=ws_s, stream=st)
            vl = s_out["verify_len"]
        if timed:
            ev["sched"][1].record(stream)
            ev["verify"][0].record(stream)
        binding.verify(x["target"], x["base"], x["e_in"], x["w_out"], x["anchor"], d_out, vl,
                       x["temperature"], x["request_id"], args.seed, out=v_out, workspace=ws_v,
                       stream=st)
        if timed:
            ev["verify"][1].record(stream)

    for _ in range(args.warmup):
        step(inp)
    torch.cuda.synchronize()
    vl_host = s_out["verify_len"].cpu().numpy() if w.scheduler else np.full(B, G)
    positions = int(vl_host.sum())
    n_rej = int((v_out["accept_len"] < (s_out["verify_len"] if w.scheduler else G)).sum().item())
    # measured acceptance: accepted tests over tests (a request stops testing at
    # its first rejection)
    acc_h = v_out["accept_len"].cpu().numpy()
    n_tests = int(np.minimum(acc_h + 1, vl_host).sum())
    acceptance = float(acc_h.sum()) / max(1, n_tests)

    # per-call timing (events around each call), then the whole-step timing
    for _ in range(max(3, min(args.steps, 20))):
        step(inp, timed=True)
        torch.cuda.synchronize()
        for k in ev:
            call_ms[k].append(ev[k][0].elapsed_time(ev[k][1]))

    # The timed rounds replay one CUDA graph of the round (its launches and
    # flag clears, captured once on a side stream): the same kernels on the
    # same resident buffers, without the per-launch gaps of eager issue.
    graph = None
    if not args.no_graph:
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap):
            step(inp, st=cap)
        stream.wait_stream(cap)
        graph.replay()
        torch.cuda.synchronize()

    clocks = ClockSampler(dev.index)
    if rank == 0:
        clocks.start()
        time.sleep(0.3)
    _barrier(world)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    h0 = time.monotonic()
    t0.record(stream)
    for _ in range(args.steps):
        if graph is not None:
            graph.replay()
        else:
            step(inp)
    t1.record(stream)
    torch.cuda.synchronize()
    h1 = time.monotonic()
    _barrier(world)
    ms = t0.elapsed_time(t1) / args.steps
    clk = clocks.stop(region=(h0, h1)) if rank == 0 else None
    # every call of the timed region must have completed cleanly: no invalid
    # input and no bounded wait that ran out
    flags = dict(draft=binding.read_device_flags(ws_d), verify=binding.read_device_flags(ws_v))
    if any(flags.values()):
        raise RuntimeError("device flags raised in the timed region: %s" % flags)
    # the spread of single rounds: a separate pass after the timed region, one
    # event pair around each round (events recorded back to back, no sync)
    n_spread = min(args.steps, 100)
    sp_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(n_spread)]
    for a, b in sp_ev:
        a.record(stream)
        if graph is not None:
            graph.replay()
        else:
            step(inp)
        b.record(stream)
    torch.cuda.synchronize()
    per_step = sorted(a.elapsed_time(b) for a, b in sp_ev)

    def _pct(q):
        return per_step[min(len(per_step) - 1, int(q * len(per_step)))]

    step_spread = dict(n=n_spread, min=per_step[0], p10=_pct(0.1), median=_pct(0.5), p90=_pct(0.9),
                       max=per_step[-1],
                       note="ms per round, one event pair around each round, a pass after the timed region")
    ms_max = _max_over_ranks(ms, world)
    total_positions = _sum_over_ranks(positions, world)
    value = total_positions / (ms_max / 1000.0)

    # the recurrent head's draft call on the same base logits (scope row f3;
    # outside the timed step, which is the Markov head's round)
    rnn_ms = None
    if w.dtype == "bf16":
        from speculative_decoding_draft_head_gb300.synth import make_rnn_head
        head = make_rnn_head(w, args.seed + rank, device=dev)
        ws_r = binding.default_workspace(binding.WS_DRAFT_RNN, B, G, V, r, dev)
        r_out = {k: torch.empty_like(t) for k, t in d_out.items()}
        e_r0, e_r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        samples = []
        for i in range(3 + max(3, min(args.steps, 20))):
            e_r0.record(stream)
            binding.draft_sample_rnn(inp["base"], head["e_in"], head["w_h"], head["w_out"], inp["anchor"],
                                     inp["temperature"], inp["request_id"], args.seed, out=r_out,
                                     workspace=ws_r, stream=stream)
            e_r1.record(stream)
            torch.cuda.synchronize()
            if i >= 3:
                samples.append(e_r0.elapsed_time(e_r1))
        rnn_ms = statistics.median(samples)
        del head

    # End to end: every step's inputs come from pinned host memory and the
    # emitted tokens go back.  The base logits and the small per-request inputs
    # are copied whole (double-buffered: step i + 1's copies run on a copy
    # stream while step i computes); of the target logits only the rows the
    # scheduler admitted, rows 0 .. L_b of each request, cross the host link:
    # dspark_pack_target gathers them from host memory on the device after the
    # schedule, and verification reads the packed rows.  The host link (about
    # 210 GB/s, copy engine or kernel reads alike) is the bound.
    per_round = ("base", "anchor", "temperature", "request_id", "conf_logits")
    host = {k: inp[k].cpu().pin_memory() for k in per_round}
    host_target = inp["target"].cpu().pin_memory()
    out_host = dict(out_tokens=torch.empty((B, G + 1), dtype=torch.int32).pin_memory(),
                    num_out=torch.empty((B,), dtype=torch.int32).pin_memory())
    target_rows = int((np.asarray(vl_host) + 1).sum()) if w.scheduler else B * (G + 1)
    h2d = sum(host[k].numel() * host[k].element_size() for k in per_round) + \
        target_rows * V * host_target.element_size()
    d2h = sum(t.numel() * t.element_size() for t in out_host.values())
    pk_out = dict(target=torch.empty((B * (G + 1), V), dtype=host_target.dtype, device=dev),
                  row0=torch.empty((B,), dtype=torch.int64, device=dev),
                  n_rows=torch.empty((1,), dtype=torch.int64, device=dev))
    vl_full = torch.full((B,), G, dtype=torch.int32, device=dev)

    def step_e2e(x):
        binding.draft_sample(x["base"], x["e_in"], x["w_out"], x["anchor"], x["temperature"],
                             x["request_id"], args.seed, out=d_out, workspace=ws_d, stream=stream)
        vl = vl_full
        if w.scheduler:
            binding.schedule_prefix(x["conf_logits"], x["pos_temp"], x["sps"], w.L_min, G, out=s_out,
                                    workspace=ws_s, stream=stream)
            vl = s_out["verify_len"]
        binding.pack_target(host_target, vl, out=pk_out, stream=stream)
        binding.verify(pk_out["target"], x["base"], x["e_in"], x["w_out"], x["anchor"], d_out, vl,
                       x["temperature"], x["request_id"], args.seed, target_row0=pk_out["row0"], out=v_out,
                       workspace=ws_v, stream=stream)

    copy_stream = torch.cuda.Stream(dev)
    bufs = [{k: (inp[k].clone() if k in per_round else inp[k]) for k in inp} for _ in range(2)]
    ev_copied = [torch.cuda.Event() for _ in range(2)]
    ev_used = [torch.cuda.Event() for _ in range(2)]
    used_recorded = [False, False]

    def issue_copy(i, start_ev=None):
        b = i % 2
        with torch.cuda.stream(copy_stream):
            if start_ev is not None:
                copy_stream.wait_event(start_ev)
            if used_recorded[b]:
                copy_stream.wait_event(ev_used[b])  # step i - 2 is done with this buffer
            for k in per_round:
                bufs[b][k].copy_(host[k], non_blocking=True)
            ev_copied[b].record(copy_stream)

    def e2e_run(n, start_ev=None):
        issue_copy(0, start_ev)
        for i in range(n):
            if i + 1 < n:
                issue_copy(i + 1)
            b = i % 2
            stream.wait_event(ev_copied[b])
            step_e2e(bufs[b])
            ev_used[b].record(stream)
            used_recorded[b] = True
            out_host["out_tokens"].copy_(v_out["out_tokens"], non_blocking=True)
            out_host["num_out"].copy_(v_out["num_out"], non_blocking=True)

    e2e_run(2)
    torch.cuda.synchronize()
    e_steps = max(3, args.steps // 4)
    _barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_run(e_steps, start_ev=e0)
    e1.record(stream)
    torch.cuda.synchronize()
    _barrier(world)
    e_ms = _max_over_ranks(e0.elapsed_time(e1) / e_steps, world)
    e_value = total_positions / (e_ms / 1000.0)

    # the device's Philox4x32-10 rate with the draft's own word code (the ALU
    # roof of the per-token draw), measured here on this GPU
    philox_peak = max(binding.selftest_philox_rate(2048) for _ in range(3))

    if rank != 0:
        return
    peaks = _peaks()
    # algorithmic bytes of one round
    draft_bytes = B * G * V * s_ + r * V * s_ + B * G * r * s_
    verify_bytes = int((vl_host + 1).sum()) * V * s_
    residual_bytes = n_rej * V * s_ * 2
    round_bytes = draft_bytes + verify_bytes + residual_bytes
    d_ms = statistics.median(call_ms["draft"])
    v_ms = statistics.median(call_ms["verify"])
    s_ms = statistics.median(call_ms["sched"])
    dominant = "draft" if d_ms >= v_ms else "verify"
    # the bf16 draft runs one launch for all positions (+ finalize); fp32 weights
    # take the SIMT kernel: one launch pair per position, or one launch for all
    # positions when a single vocabulary segment covers each row
    launches_draft = 2 if w.dtype == "bf16" else _simt_draft_launches(B, G, V)
    dom_bytes = draft_bytes if dominant == "draft" else verify_bytes + residual_bytes
    dom_ms = d_ms if dominant == "draft" else v_ms
    # draft: one (cooperative) launch of the Markov-head kernel for all block
    # positions + one finalize; verify: rows, decide, final draw, merge
    launches_per_call = 2 if dominant == "draft" else 4
    achieved = dom_bytes / (dom_ms / 1000.0) / 1e9
    bias_flops = 2.0 * B * G * V * r
    traffic = _read_traffic(w, dominant)
    # the ALU roof: one Philox4x32-10 block per four tokens of a draw; the
    # draft draws B G V tokens, the final draw of verification one row per
    # request (B V)
    draft_blocks = B * G * ((V + 3) // 4)
    final_blocks = B * ((V + 3) // 4)

    def roof(nbytes, blocks, ms_call, dram=None):
        t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
        t_alu = blocks / philox_peak
        hbm = dict(achieved=nbytes / (ms_call / 1000.0) / 1e9, peak=peaks["hbm_gbs"], unit="GB/s",
                   frac=nbytes / (ms_call / 1000.0) / 1e9 / peaks["hbm_gbs"], floor_us=t_hbm * 1e6)
        alu = dict(achieved=blocks / (ms_call / 1000.0) / 1e9, peak=philox_peak / 1e9,
                   unit="G Philox4x32-10 blocks/s", frac=blocks / (ms_call / 1000.0) / philox_peak,
                   floor_us=t_alu * 1e6)
        return dict(bound="alu" if t_alu > t_hbm else "hbm", hbm=hbm, alu=alu)

    r_draft = roof(draft_bytes, draft_blocks, d_ms)
    r_verify = roof(verify_bytes + residual_bytes, final_blocks, v_ms)
    r_dom = r_draft if dominant == "draft" else r_verify
    dom_roof = r_dom[r_dom["bound"]]
    line = dict(
        metric=METRIC, value=value, unit=UNIT, n_gpus=world, steps=args.steps, warmup=args.warmup,
        ms_per_step=ms_max, higher_is_better=True, scaling="weak", vs_baseline=None, dtype="f32",
        data="synthetic", config=_config(w),
        hbm_gbs=round_bytes / (ms / 1000.0) / 1e9,
        positions_per_step=positions,
        drafted_positions_per_s=B * G / (d_ms / 1000.0),
        acceptance=dict(accepted_over_tested=acceptance, tests=n_tests,
                        note="per-test acceptance min(1, p/q) realised on the synthetic workload"),
        roofline=dict(bound=r_dom["bound"], achieved=dom_roof["achieved"], peak=dom_roof["peak"],
                      unit=dom_roof["unit"], frac=dom_roof["frac"], traffic=traffic,
                      kernel=("draft call: markov_tc_kernel (all %d positions, one launch) + finalize" % G
                              if dominant == "draft" else "verify call (%d launches)" % launches_per_call),
                      peak_source=("measured live: dspark_selftest_philox_rate (the draft's Philox code, "
                                   "2048 threads per SM), best of 3" if r_dom["bound"] == "alu" else
                                   peaks["source"] + " (MEASURED_PEAKS.json hbm_gbs)"),
                      hbm_frac=r_dom["hbm"]["frac"], alu_frac=r_dom["alu"]["frac"],
                      dram_gbs=(None if traffic is None else traffic / (dom_ms / 1000.0) / 1e9)),
        rooflines=dict(draft=r_draft, verify=r_verify,
                       note="per call (events around the call, eager issue): hbm = algorithmic bytes "
                            "over the call time against the measured copy bandwidth; alu = Philox "
                            "blocks (one per four drawn tokens) over the call time against the "
                            "device's measured Philox rate; bound = the roof with the longer floor"),
        step_ms=step_spread,
        calls_ms=dict(draft=d_ms, schedule=s_ms, verify=v_ms),
        step_order=("draft, schedule, verify on one stream" +
                    (", replayed from one CUDA graph (calls_ms timed eagerly)" if graph is not None else "")),
        rnn_head=(None if rnn_ms is None else
                  dict(draft_ms=rnn_ms, launches=2 * G + 1,
                       note="recurrent-head draft call (state update + tensor-core draw per position, "
                            "then finalize), not part of the timed round")),
        bias_gemm=dict(flops_per_round=bias_flops,
                       tflops_over_draft_time=bias_flops / (d_ms / 1000.0) / 1e12,
                       peak_tflops=peaks["bf16_tflops_sustained"]),
        e2e=dict(value=e_value, unit=UNIT, h2d_bytes_per_step=int(h2d), d2h_bytes_per_step=int(d2h),
                 ms_per_step=e_ms,
                 copies="every step from pinned host memory: base logits and per-request inputs copied "
                        "whole (overlapped with the previous step, two buffers, a copy stream); target "
                        "logits only for the scheduled rows 0..L_b of each request (%d of %d rows), "
                        "gathered on the device by dspark_pack_target" % (target_rows, B * (G + 1))),
        gpu_launches=args.steps * (launches_draft + (1 if w.scheduler else 0) + 4),
        device_flags=flags,
        clocks=clk,
    )
    if not args.no_cpu_baseline and world == 1:
        h = {k: t.cpu() for k, t in inp.items()}
        line["cpu_baseline"] = cpu_baseline_line(w, h, args.seed, args.cpu_budget)
    print(json.dumps(line))


def _simt_draft_launches(B, G, V):
    """Launches of a draft call with fp32 weights: one per position and its
    finalize, or a single launch for all positions when one vocabulary
    segment covers each row (the library's SIMT plan: 8 requests per block,
    about two blocks per SM, segments of at least 1024 tokens)."""
    row_blocks = (B + 7) // 8
    nsplit = max(1, min((2 * 152 + row_blocks - 1) // row_blocks, (V + 1023) // 1024))
    return 1 if nsplit == 1 else 2 * G


def _read_traffic(w, kernel):
    """DRAM bytes per launch from the committed ncu summary, if one matches."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get("%s/%s" % (w.name, kernel))
    return None if e is None else e.get("dram_bytes_per_call")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    # about a tenth of a second of timed rounds: several clock samples (every
    # 25 ms) fall inside it
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="dspark5")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="issue the timed rounds' calls eagerly instead of replaying a CUDA graph of the round")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    from speculative_decoding_draft_head_gb300.synth import WORKLOADS
    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()

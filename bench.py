#!/usr/bin/env python3
"""Benchmark of libgdn on GB300: one JSON line on rank 0.

Workloads (synthetic, seeded; see gated_deltanet_mixer_gb300/inputs.py):
  prefill  Qwen3.5-4B-shaped GDN layer: B=4, T=8192, Hk=16, Hv=32, Dk=Dv=128,
           bf16 io, fp32 state.  `value` = prefill tokens/s over all ranks.
  decode   Qwen3.8-27B-shaped batched decode: B=256, Hk=16, Hv=48; one bench
           step = 64 consecutive gdn_decode_step calls.  Reported under
           "decode" as state GB/s and total GB/s against HBM.

  next     the extended calls, per GPU, under "next": the 4B prefill with
           the gates formed from raw projections, a packed batch of 24
           sequences (log-uniform lengths 100..4000), and 4-token decoding
           from the cache at the 27B decode shape with and without per-token
           state snapshots; and the 27B in_proj / out_proj projections
           (gdn_linear, 8192 tokens) against the bf16 tensor peak.

--impl reference times the fp64 CPU oracle instead, on a bounded sample of the
same prefill workload, with the same metric and unit.

Multi-GPU (torchrun): every rank runs its own full prefill batch (weak
scaling, no collective on the data path); the max over ranks of the timed
region sets the time.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GDN prefill tokens/s (4B/27B shapes) + decode state GB/s vs HBM peak, 1×GB300"
D = 128
PREFILL_KERNELS_PER_CALL = 3   # gdn_prefill_ex with a full workspace: q^/k^, the chunk-parallel prep, the sequential pass
DECODE_KERNELS_PER_CALL = 1    # gdn_decode_step launches one kernel
DECODE_CALLS_PER_STEP = 64
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ------------------------------------------------------------ work counts
def conv_channels(Hk, Hv):
    return (2 * Hk + Hv) * D


def prefill_bytes(B, T, Hk, Hv, io=2):
    """Algorithmic HBM bytes of one prefill call: every input read once,
    every output written once."""
    C = conv_channels(Hk, Hv)
    per_token = io * C + 2 * io * Hv * D + 8 * Hv          # qkv, z, o, g+beta
    per_seq = 2 * Hv * D * D * 4 + 2 * 3 * C * io          # S0 + S_T, conv0 + conv_T
    weights = C * 4 * io + D * io
    return B * T * per_token + B * per_seq + weights


def prefill_flops(B, T, Hk, Hv, chunk=64):
    """Dense-contraction flops of the chunked (WY) form per call: per key
    head Q K^T and K K^T; per value head U, W, the masked (QK^T) Delta, and
    the three state products W S, Q S, K^T Delta."""
    per_token = Hk * 4 * chunk * D + Hv * (3 * 2 * chunk * D + 6 * D * D)
    return B * T * per_token


def decode_bytes(B, Hk, Hv, io=2):
    """Algorithmic HBM bytes of one decode call."""
    C = conv_channels(Hk, Hv)
    per_seq = 8 * Hv * D * D + 2 * 3 * C * io + io * C + 2 * io * Hv * D + 8 * Hv
    return B * per_seq + C * 4 * io + D * io


def decode_state_bytes(B, Hv):
    return B * 8 * Hv * D * D


def packed_bytes(lengths, Hk, Hv, io=2, raw_gates=False):
    """Algorithmic HBM bytes of one packed prefill call."""
    C = conv_channels(Hk, Hv)
    N, B = sum(lengths), len(lengths)
    gates = 2 * io * Hv if raw_gates else 8 * Hv
    per_token = io * C + 2 * io * Hv * D + gates
    per_seq = 2 * Hv * D * D * 4 + 2 * 3 * C * io
    return N * per_token + B * per_seq + C * 4 * io + D * io + (B + 1) * 4 + (8 * Hv if raw_gates else 0)


def decode_multi_bytes(B, T, Hk, Hv, io=2, snapshots=True):
    """Algorithmic HBM bytes of one T-token decode call: the state read and
    written once, one snapshot per token, the window in and out, the tokens."""
    C = conv_channels(Hk, Hv)
    per_seq = 8 * Hv * D * D + (4 * T * Hv * D * D if snapshots else 0) + 2 * 3 * C * io \
        + T * (io * C + 2 * io * Hv * D + 8 * Hv)
    return B * per_seq + C * 4 * io + D * io


WORKLOAD_LABEL = {
    "4b_prefill": "Qwen3.5-4B-shaped GDN layer prefill",
    "0.8b_prefill": "Qwen3.5-0.8B-shaped GDN layer prefill",
    "27b_prefill": "Qwen3.8-27B-shaped GDN long prefill",
}
# What the path computes in: io is bf16, the tensor-core operands fp16 (the
# state path's as hi/lo pairs), the state and every accumulation fp32.
DTYPE = "bf16 io, fp16 MMA operands (hi/lo pairs on the state path), fp32 state and accumulation"


def workload_name(name, p):
    return "%s: B=%d, T=%d, Hk=%d, Hv=%d, Dk=Dv=128, bf16 io, fp32 state" % (
        WORKLOAD_LABEL[name], p.B, p.T, p.Hk, p.Hv)


# Packed-batch length mix: 24 sequences, log-uniform lengths in [100, 4000]
# (a serving batch of prompts), seed 7.
def varlen_lengths():
    gen = np.random.Generator(np.random.PCG64(7))
    return [int(round(x)) for x in np.exp(gen.uniform(np.log(100.0), np.log(4000.0), size=24))]


# ----------------------------------------------------------------- helpers
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return {k: float(pk[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def source_sha(relpath):
    with open(os.path.join(ROOT, relpath), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def recorded_traffic(kernel_key, source_relpaths):
    """DRAM bytes per launch recorded from an ncu capture, if every source it
    depends on is unchanged since; otherwise None."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(kernel_key)
    except (OSError, ValueError):
        return None
    if not rec:
        return None
    shas = rec.get("sources_sha256", {})
    if sorted(shas) != sorted(source_relpaths) or any(shas[p] != source_sha(p) for p in source_relpaths):
        return None
    return rec.get("dram_bytes_per_launch")


def bind_gpu_local_cpus(uuid):
    """Run this process on the CPUs the GPU's PCI device reports as local (its
    NUMA node), where they are among those allowed, so that the pinned host
    buffers of the end-to-end measurement are allocated next to the GPU, as a
    serving process would place them.  Returns the CPUs used, or None where
    the topology is not readable (nothing is changed then)."""
    try:
        cmd = ["nvidia-smi", "--query-gpu=pci.bus_id", "--format=csv,noheader"] + (["-i", uuid] if uuid else [])
        bus = subprocess.check_output(cmd, text=True, stderr=subprocess.DEVNULL).strip().splitlines()[0]
        dom, rest = bus.split(":", 1)  # "00000009:01:00.0" -> "0009:01:00.0"
        with open("/sys/bus/pci/devices/%04x:%s/local_cpulist" % (int(dom, 16), rest.lower())) as f:
            text = f.read().strip()
        local = set()
        for part in text.split(","):
            lo, _, hi = part.partition("-")
            local.update(range(int(lo), int(hi or lo) + 1))
        use = local & os.sched_getaffinity(0)
        if not use:
            return None
        if use != os.sched_getaffinity(0):
            os.sched_setaffinity(0, use)
        return sorted(use)
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 50 ms."""
    QUERY = ("index,uuid,utilization.gpu,clocks.sm,clocks.max.sm,power.draw,"
             "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid=None):
        self.uuid = uuid
        self.proc = None
        self.file = None

    def start(self):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        cmd = ["nvidia-smi", "--query-gpu=" + self.QUERY, "--format=csv,noheader,nounits",
               "-lms", "50"]
        if self.uuid:
            cmd += ["-i", self.uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [ln.split(", ") for ln in self.file.read().splitlines() if ln.strip()]
        self.file.close()
        os.unlink(self.file.name)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        load, reasons, maxes = [], set(), []
        for r in rows:
            if len(r) < 11:
                continue
            try:
                util, sm, smax = float(r[2]), float(r[3]), float(r[4])
            except ValueError:
                continue
            maxes.append(smax)
            if util >= 50:
                load.append(sm)
                for n, v in zip(names, r[7:11]):
                    if v.strip().lower() == "active":
                        reasons.add(n)
        return {"sm_mhz": statistics.median(load) if load else None,
                "sm_max_mhz": max(maxes) if maxes else None,
                "reasons": sorted(reasons), "samples_under_load": len(load),
                "samples": len(rows)}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def rank_case(case, rank):
    """Input seed of `case` on `rank`: every rank draws its own batch."""
    return case + 1000 * rank


def max_over_ranks(x, world, device="cuda"):
    """The largest of every rank's `x` (a time in ms); `x` itself at world 1."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------- oracle timing
def oracle_run(p, n_tok, threads):
    """The oracle, as it stands, on the workload's first `n_tok` tokens: whole
    sequences first (all value heads), then a prefix of the next.  Seconds."""
    from oracle import oracle as O

    a = p.arrays
    nb, rem = divmod(n_tok, p.T)
    t0 = time.perf_counter()
    for b0, b1, T in ((0, nb, p.T), (nb, nb + 1, rem)):
        if b1 <= b0 or T == 0:
            continue
        O.gdn_prefill(a["qkv_pre"][b0:b1, :T], a["z"][b0:b1, :T], a["g"][b0:b1, :T],
                      a["beta"][b0:b1, :T], a["conv_w"], a["norm_w"],
                      None if a["S0"] is None else a["S0"][b0:b1],
                      None if a["conv0"] is None else a["conv0"][b0:b1], Hk=p.Hk, Hv=p.Hv,
                      threads=threads, want_conv=False)
    return time.perf_counter() - t0


def oracle_tokens_per_s(p, budget_s, threads):
    """Size a sample to about `budget_s` seconds of oracle work (capped at the
    whole workload) and time it.  Returns (tokens, seconds)."""
    probe = min(p.T, 256)
    rate = probe / max(oracle_run(p, probe, threads), 1e-6)
    n = int(max(probe, min(p.B * p.T, rate * budget_s)))
    return n, oracle_run(p, n, threads)


# --------------------------------------------------------------- GPU arm
def gdn_arm(args, world, rank, local):
    import torch

    from gated_deltanet_mixer_gb300 import build as gdn_build
    from gated_deltanet_mixer_gb300 import gdn
    from gated_deltanet_mixer_gb300 import inputs as I

    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    gdn_build.build()
    gdn.lib()
    peaks, peak_src = load_peaks()

    # ---- prefill inputs (each rank its own batch)
    spec = dict(I.CASES[args.workload])
    spec["case"] = rank_case(spec["case"], rank)
    p = I.prefill_problem(**spec)
    t_io = torch.bfloat16 if p.io == "bf16" else torch.float32
    a = p.arrays

    def dev(x, dt=torch.float32):
        return None if x is None else torch.from_numpy(x).to("cuda").to(dt)

    x = dict(qkv_pre=dev(a["qkv_pre"], t_io), z=dev(a["z"], t_io), g=dev(a["g"]),
             beta=dev(a["beta"]), conv_w=dev(a["conv_w"], t_io), norm_w=dev(a["norm_w"], t_io),
             S0=dev(a["S0"]), conv0=dev(a["conv0"], t_io))
    o, S_T, conv_T = gdn.alloc_prefill_outputs(p.B, p.T, p.Hk, p.Hv, t_io)
    stream = torch.cuda.current_stream()

    # The chunk-parallel path: the workspace holds q^ and k^ of every token and
    # key head and every chunk's state-independent part between the call's
    # three kernels (calls run one after another on the stream, so one
    # workspace serves them all).
    ws = torch.empty(gdn.gdn_prefill_workspace_bytes(p.B, p.T, p.Hk, p.Hv), dtype=torch.uint8, device="cuda")

    def prefill_call(xx, oo, ss, cc):
        gdn.gdn_prefill_ex(xx["qkv_pre"], xx["z"], xx["g"], xx["beta"], xx["conv_w"], xx["norm_w"],
                           xx["S0"], xx["conv0"], oo, ss, cc, Hk=p.Hk, Hv=p.Hv, workspace=ws, stream=stream)

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(local).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        uuid = None
    host_cpus = bind_gpu_local_cpus(uuid)
    clocks = ClockSampler(uuid)
    clocks.start()

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        prefill_call(x, o, S_T, conv_T)
    barrier()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    t_beg, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_beg.record(stream)
    for k in range(args.steps):
        ev[k][0].record(stream)
        prefill_call(x, o, S_T, conv_T)
        ev[k][1].record(stream)
    t_end.record(stream)
    barrier()
    if gdn.gdn_device_status(stream) != 0:
        raise RuntimeError("device status not OK after the prefill timing")
    total_ms = t_beg.elapsed_time(t_end)
    launch_ms = float(np.mean([s.elapsed_time(e) for s, e in ev]))
    total_ms = max_over_ranks(total_ms, world)
    ms_per_step = total_ms / args.steps
    tokens = p.B * p.T
    value = world * tokens / (ms_per_step * 1e-3)

    # ---- decode: 64 consecutive calls per step, inputs resident
    dec = None
    if not args.no_decode:
        dp = I.decode_problem(**dict(I.DECODE_CASE, case=rank_case(I.DECODE_CASE["case"], rank)))
        S = dev(dp.S)
        conv = [dev(dp.conv, t_io), dev(dp.conv, t_io)]
        cw, nw = dev(dp.conv_w, t_io), dev(dp.norm_w, t_io)
        q_all = dev(dp.qkv_pre, t_io)
        z_all = dev(dp.z, t_io)
        g_all, b_all = dev(dp.g), dev(dp.beta)
        od = torch.empty(dp.B, dp.Hv * D, device="cuda", dtype=t_io)

        def decode_step_block():
            for s in range(DECODE_CALLS_PER_STEP):
                gdn.gdn_decode_step(q_all[s], z_all[s], g_all[s], b_all[s], cw, nw, S,
                                    conv[s % 2], conv[(s + 1) % 2], od, Hk=dp.Hk, Hv=dp.Hv,
                                    stream=stream)

        for _ in range(args.warmup):
            decode_step_block()
        barrier()
        d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        d0.record(stream)
        for _ in range(args.steps):
            decode_step_block()
        d1.record(stream)
        barrier()
        if gdn.gdn_device_status(stream) != 0:
            raise RuntimeError("device status not OK after the decode timing")
        dec_ms = d0.elapsed_time(d1)
        dec_ms = max_over_ranks(dec_ms, world)
        call_ms = dec_ms / (args.steps * DECODE_CALLS_PER_STEP)
        dbytes = decode_bytes(dp.B, dp.Hk, dp.Hv)
        sbytes = decode_state_bytes(dp.B, dp.Hv)
        dach = dbytes / (call_ms * 1e-3) / 1e9
        dec = {
            "workload": "Qwen3.8-27B-shaped GDN decode: B=256 sequences x 1 token, Hk=16, Hv=48, "
                        "Dk=Dv=128, bf16 io, fp32 state; one step = 64 consecutive calls",
            "value": world * sbytes / (call_ms * 1e-3) / 1e9, "unit": "state GB/s",
            "total_gbs": world * dach, "ms_per_call": call_ms,
            "ms_per_step": dec_ms / args.steps,
            "tokens_per_s": world * dp.B / (call_ms * 1e-3),
            "gpu_launches": args.steps * DECODE_CALLS_PER_STEP * DECODE_KERNELS_PER_CALL,
            "roofline": {"bound": "hbm", "achieved": dach, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": dach / peaks["hbm_gbs"],
                         "traffic": recorded_traffic("decode_kernel", DECODE_SOURCES),
                         "algorithmic_bytes_per_launch": dbytes,
                         "peak_source": peak_src + " hbm_gbs (burst copy)"},
        }
        del S, conv, q_all, z_all, g_all, b_all, od
    # ---- the other prefill shapes of the metric (0.8B, 27B), one call each
    shapes = None if args.no_shapes else shape_rows(args, peaks, peak_src, stream, barrier, world, rank)
    # ---- the extended calls: raw gates, packed batch, multi-token decode
    nxt = None if args.no_next else next_rows(args, x, o, S_T, conv_T, p, peaks, peak_src, stream,
                                              barrier, world, rank)
    clk = clocks.stop()

    # ---- end to end through the public API with host buffers
    pin = {k: (None if v is None else v.cpu().pin_memory()) for k, v in x.items()}
    ho = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    hS = torch.empty(S_T.shape, dtype=S_T.dtype).pin_memory()
    hc = torch.empty(conv_T.shape, dtype=conv_T.dtype).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in pin.values() if v is not None)
    d2h = sum(t.numel() * t.element_size() for t in (ho, hS, hc))
    e2e_steps = max(3, min(args.steps, 8))
    # Pipelined as a serving loop would run it: two device buffer sets; step
    # k's host->device copies (stream s_in) and step k-1's device->host copies
    # (s_out) overlap step k-1's / k's call (the compute stream), ordered by
    # events.  Every step still moves all its inputs and outputs.
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    xs = [x, {k: (None if v is None else torch.empty_like(v)) for k, v in x.items()}]
    outs = [(o, S_T, conv_T), tuple(torch.empty_like(t) for t in (o, S_T, conv_T))]
    hos = [(ho, hS, hc), tuple(torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (o, S_T, conv_T))]
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    used = [False, False]

    def e2e_step(k):
        bsel = k % 2
        if used[bsel]:
            s_in.wait_event(ev_comp[bsel])  # the call that read these inputs is done
        with torch.cuda.stream(s_in):
            for key, v in pin.items():
                if v is not None:
                    xs[bsel][key].copy_(v, non_blocking=True)
        ev_in[bsel].record(s_in)
        stream.wait_event(ev_in[bsel])
        if used[bsel]:
            stream.wait_event(ev_out[bsel])  # these outputs were read back
        prefill_call(xs[bsel], *outs[bsel])
        ev_comp[bsel].record(stream)
        s_out.wait_event(ev_comp[bsel])
        with torch.cuda.stream(s_out):
            for hbuf, dbuf in zip(hos[bsel], outs[bsel]):
                hbuf.copy_(dbuf, non_blocking=True)
        ev_out[bsel].record(s_out)
        used[bsel] = True

    # two untimed repetitions (on some hosts the first passes over freshly
    # pinned buffers run several times slower), then three timed ones; the
    # median is reported
    for k in range(2 * e2e_steps):
        e2e_step(k)
    barrier()
    e2e_reps = []
    for _ in range(3):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s_in)
        for k in range(e2e_steps):
            e2e_step(k)
        e1.record(s_out)
        barrier()
        e2e_reps.append(max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world))
    e2e_ms = statistics.median(e2e_reps)

    # ---- roofline of the prefill kernel
    pbytes = prefill_bytes(p.B, p.T, p.Hk, p.Hv, 2 if p.io == "bf16" else 4)
    pflops = prefill_flops(p.B, p.T, p.Hk, p.Hv)
    ach = pbytes / (launch_ms * 1e-3) / 1e9
    tfl = pflops / (launch_ms * 1e-3) / 1e12
    result = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": DTYPE, "data": "synthetic (seeded; model-shaped random inputs, no weights needed)",
        "config": {"workload": workload_name(args.workload, p),
                   "io_dtype": p.io, "state_dtype": "f32",
                   "l2": "inputs larger than L2 (%.2f GB read+written per step; L2 129 MB)"
                         % (pbytes / 1e9),
                   "parallelism": "one GPU per rank, each rank its own batch (weak scaling)"},
        "roofline": {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": ach / peaks["hbm_gbs"],
                     "traffic": recorded_traffic("prefill_call_4b", PREFILL_SOURCES),
                     "algorithmic_bytes_per_launch": pbytes, "launch_ms": launch_ms,
                     "scope": "one gdn_prefill_ex call: prefill_qk_kernel (q^, k^ once per key head), "
                              "prefill_prep_kernel (every chunk's T, U, W, M at once), prefill_seq_kernel "
                              "(the state recurrence per sequence and value head); the mixer's algorithmic "
                              "bytes over the call's device time; traffic counts the workspace round trip",
                     "peak_source": peak_src + " hbm_gbs (burst copy)"},
        "roofline_tensor": {"bound": "tensor", "achieved": tfl, "peak": peaks["bf16_tflops"],
                            "unit": "TFLOP/s", "frac": tfl / peaks["bf16_tflops"],
                            "algorithmic_flops_per_launch": pflops,
                            "peak_source": peak_src + " bf16_tflops (burst)"},
        "e2e": {"value": world * tokens / (e2e_ms * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "ms_per_step_reps": e2e_reps, "steps_per_rep": e2e_steps,
                "host_cpus": ("%d GPU-local CPUs" % len(host_cpus)) if host_cpus else "as scheduled",
                "pipelined": "two buffer sets: a step's copies overlap the neighbouring steps' calls"},
        "gpu_launches": args.steps * PREFILL_KERNELS_PER_CALL,
        "clocks": clk,
        "decode": dec,
        "prefill_shapes": shapes,
        "next": nxt,
    }
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    # ---- CPU baseline: the oracle as it stands, rank 0, single GPU only
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        from oracle import oracle as O
        threads = O.default_threads()
        T_s, secs = oracle_tokens_per_s(p, args.cpu_budget, threads)
        result["cpu_baseline"] = {
            "value": T_s / secs, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": "fp64 oracle on the first %d of the workload's %d tokens (%d sequences "
                      "x %d), all %d value heads, %.1f s" % (T_s, p.B * p.T, p.B, p.T, p.Hv, secs)}
    if rank == 0:
        print(json.dumps(result))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# The sources a recorded prefill / decode traffic figure depends on.
PREFILL_SOURCES = ["gated_deltanet_mixer_gb300/csrc/prefill_split.cu",
                   "gated_deltanet_mixer_gb300/csrc/prefill_chunked.cu",
                   "gated_deltanet_mixer_gb300/csrc/chunk_math.cuh"]
DECODE_SOURCES = ["gated_deltanet_mixer_gb300/csrc/decode.cu"]


def time_launches(fn, steps, warmup, stream, barrier, world=1):
    """Mean device ms per call of fn (one library call), CUDA events on
    `stream`; the largest over the ranks."""
    import torch
    for _ in range(warmup):
        fn()
    barrier()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for k in range(steps):
        ev[k][0].record(stream)
        fn()
        ev[k][1].record(stream)
    barrier()
    return max_over_ranks(float(np.mean([s.elapsed_time(e) for s, e in ev])), world)


def split_overlaps(B, Hv):
    """Whether a fixed-length call with a full workspace runs both parts of
    the chunk-parallel prefill in one cooperative launch (prefill_qk_kernel +
    prefill_overlap_kernel) rather than three kernels: at most half as many
    (sequence, value head) units as SMs."""
    import torch
    return 2 * B * Hv <= torch.cuda.get_device_properties(0).multi_processor_count


def shape_rows(args, peaks, peak_src, stream, barrier, world, rank):
    """The prefill shapes the metric names besides the main workload: one
    gdn_prefill_ex call each (the benchmarked path: a workspace given), inputs
    resident, tokens/s with the call's HBM and bf16 tensor rooflines."""
    import torch

    from gated_deltanet_mixer_gb300 import gdn
    from gated_deltanet_mixer_gb300 import inputs as I

    out = {}
    for name in ("0.8b_prefill", "27b_prefill"):
        if name == args.workload:
            continue
        spec = dict(I.CASES[name])
        spec["case"] = rank_case(spec["case"], rank)
        q = I.prefill_problem(**spec)
        a = q.arrays
        bf = torch.bfloat16

        def dev(v, dt=torch.float32):
            return None if v is None else torch.from_numpy(v).to("cuda").to(dt)

        qx = dict(qkv_pre=dev(a["qkv_pre"], bf), z=dev(a["z"], bf), g=dev(a["g"]), beta=dev(a["beta"]),
                  conv_w=dev(a["conv_w"], bf), norm_w=dev(a["norm_w"], bf), S0=dev(a["S0"]),
                  conv0=dev(a["conv0"], bf))
        del q.arrays
        qo, qS, qc = gdn.alloc_prefill_outputs(q.B, q.T, q.Hk, q.Hv, bf)
        qws = torch.empty(gdn.gdn_prefill_workspace_bytes(q.B, q.T, q.Hk, q.Hv), dtype=torch.uint8,
                          device="cuda")
        steps = max(3, min(args.steps, 10))
        ms = time_launches(lambda: gdn.gdn_prefill_ex(
            qx["qkv_pre"], qx["z"], qx["g"], qx["beta"], qx["conv_w"], qx["norm_w"], qx["S0"], qx["conv0"],
            qo, qS, qc, Hk=q.Hk, Hv=q.Hv, workspace=qws, stream=stream), steps, args.warmup, stream, barrier,
            world)
        nb = prefill_bytes(q.B, q.T, q.Hk, q.Hv)
        fl = prefill_flops(q.B, q.T, q.Hk, q.Hv)
        ach, tf = nb / (ms * 1e-3) / 1e9, fl / (ms * 1e-3) / 1e12
        out[name] = {
            "workload": workload_name(name, q), "value": world * q.B * q.T / (ms * 1e-3),
            "unit": "tokens/s", "ms_per_launch": ms, "launches_timed": steps,
            "kernels_per_launch": 2 if split_overlaps(q.B, q.Hv) else 3,
            "roofline": {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": ach / peaks["hbm_gbs"], "algorithmic_bytes_per_launch": nb,
                         "traffic": recorded_traffic("prefill_call_" + name.split("_")[0], PREFILL_SOURCES),
                         "peak_source": peak_src + " hbm_gbs (burst copy)"},
            "roofline_tensor": {"bound": "tensor", "achieved": tf, "peak": peaks["bf16_tflops"],
                                "unit": "TFLOP/s", "frac": tf / peaks["bf16_tflops"],
                                "algorithmic_flops_per_launch": fl,
                                "peak_source": peak_src + " bf16_tflops (burst)"}}
        del qx, qo, qS, qc, qws
        torch.cuda.empty_cache()
    if gdn.gdn_device_status(stream) != 0:
        raise RuntimeError("device status not OK after the prefill shapes")
    return out


def next_rows(args, x, o, S_T, conv_T, p, peaks, peak_src, stream, barrier, world, rank):
    """Throughput of the extended entry points on model-shaped inputs (each
    input larger than L2), per GPU."""
    import torch

    from gated_deltanet_mixer_gb300 import gdn
    from gated_deltanet_mixer_gb300 import inputs as I

    def dev(a, dt=torch.float32):
        return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to("cuda").to(dt)

    bf = torch.bfloat16
    hbm = peaks["hbm_gbs"]
    out = {}
    steps = max(3, min(args.steps, 10))

    # raw gate projections on the 4B prefill workload
    rg = I.raw_gate_arrays(rank_case(60, rank), (p.B, p.T), p.Hv, "bf16")
    rgd = dict(a=dev(rg["a"], bf), b=dev(rg["b"], bf), A_log=dev(rg["A_log"]),
               dt_bias=dev(rg["dt_bias"]))
    ws = torch.empty(gdn.gdn_prefill_workspace_bytes(p.B, p.T, p.Hk, p.Hv), dtype=torch.uint8, device="cuda")
    ms = time_launches(lambda: gdn.gdn_prefill_ex(
        x["qkv_pre"], x["z"], None, None, x["conv_w"], x["norm_w"], x["S0"], x["conv0"], o, S_T,
        conv_T, Hk=p.Hk, Hv=p.Hv, raw_gates=rgd, workspace=ws, stream=stream), steps, args.warmup, stream,
        barrier, world)
    nb = packed_bytes([p.T] * p.B, p.Hk, p.Hv, raw_gates=True)
    out["prefill_raw_gates"] = {
        "workload": "4B-shaped prefill (B=%d, T=%d) with beta, g formed from raw a, b, A_log, "
                    "dt_bias inside the kernel" % (p.B, p.T),
        "value": world * p.B * p.T / (ms * 1e-3), "unit": "tokens/s", "ms_per_launch": ms,
        "roofline": {"bound": "hbm", "achieved": nb / (ms * 1e-3) / 1e9, "peak": hbm, "unit": "GB/s",
                     "frac": nb / (ms * 1e-3) / 1e9 / hbm, "peak_source": peak_src}}
    del rgd

    # packed variable-length batch at the 4B head shape
    lens = varlen_lengths()
    q = I.packed_problem(lens, p.Hk, p.Hv, io="bf16", case=rank_case(61, rank))
    qa = q.arrays
    qx = {k: dev(qa[k], bf if k in ("qkv_pre", "z", "conv_w", "norm_w", "conv0") else torch.float32)
          for k in ("qkv_pre", "z", "g", "beta", "conv_w", "norm_w", "S0", "conv0")}
    cu = torch.from_numpy(q.cu_seqlens).to("cuda")
    qo = torch.empty(q.N, p.Hv * D, device="cuda", dtype=bf)
    qS = torch.empty(len(lens), p.Hv, D, D, device="cuda")
    qc = torch.empty(len(lens), 3, q.C, device="cuda", dtype=bf)
    qws = torch.empty(gdn.gdn_prefill_workspace_bytes(len(lens), q.N, p.Hk, p.Hv, packed=True),
                      dtype=torch.uint8, device="cuda")
    ms = time_launches(lambda: gdn.gdn_prefill_ex(
        qx["qkv_pre"], qx["z"], qx["g"], qx["beta"], qx["conv_w"], qx["norm_w"], qx["S0"],
        qx["conv0"], qo, qS, qc, Hk=p.Hk, Hv=p.Hv, cu_seqlens=cu, workspace=qws, stream=stream), steps,
        args.warmup, stream, barrier, world)
    nb = packed_bytes(lens, p.Hk, p.Hv)
    out["prefill_varlen"] = {
        "workload": "packed batch of %d sequences (log-uniform lengths 100..4000, %d tokens), "
                    "Hk=%d, Hv=%d, bf16 io" % (len(lens), q.N, p.Hk, p.Hv),
        "value": world * q.N / (ms * 1e-3), "unit": "tokens/s", "ms_per_launch": ms,
        "roofline": {"bound": "hbm", "achieved": nb / (ms * 1e-3) / 1e9, "peak": hbm, "unit": "GB/s",
                     "frac": nb / (ms * 1e-3) / 1e9 / hbm, "peak_source": peak_src}}
    del qx, qo, qS, qc, cu, qws, ws

    # T-token decode from the cache (speculative verification), 27B decode shape
    T = 4
    dp = I.decode_problem(**dict(I.DECODE_CASE, steps=T, case=rank_case(I.DECODE_CASE["case"] + 70, rank)))
    S = dev(dp.S)
    snap = torch.empty(dp.B, T, dp.Hv, D, D, device="cuda")
    conv_in, conv_out = dev(dp.conv, bf), torch.empty(dp.B, 3, dp.C, device="cuda", dtype=bf)
    tq = dev(dp.qkv_pre.transpose(1, 0, 2), bf)
    tz = dev(dp.z.transpose(1, 0, 2), bf)
    tg, tb = dev(dp.g.transpose(1, 0, 2)), dev(dp.beta.transpose(1, 0, 2))
    cw, nw = dev(dp.conv_w, bf), dev(dp.norm_w, bf)
    od = torch.empty(dp.B, T, dp.Hv * D, device="cuda", dtype=bf)
    for with_snap in (True, False):
        ms = time_launches(lambda: gdn.gdn_decode_ex(
            tq, tz, tg, tb, cw, nw, S, conv_in, conv_out, od, Hk=dp.Hk, Hv=dp.Hv,
            S_snap=snap if with_snap else None, stream=stream), steps, args.warmup, stream, barrier, world)
        nb = decode_multi_bytes(dp.B, T, dp.Hk, dp.Hv, snapshots=with_snap)
        out["decode_multi%s" % ("_snapshots" if with_snap else "")] = {
            "workload": "27B-shaped decode of %d tokens per sequence from the cache, B=%d, Hv=%d%s"
                        % (T, dp.B, dp.Hv, ", state snapshot after every token" if with_snap else ""),
            "value": world * dp.B * T / (ms * 1e-3), "unit": "tokens/s", "ms_per_launch": ms,
            "roofline": {"bound": "hbm", "achieved": nb / (ms * 1e-3) / 1e9, "peak": hbm,
                         "unit": "GB/s", "frac": nb / (ms * 1e-3) / 1e9 / hbm,
                         "traffic": None if with_snap else recorded_traffic("decode_multi_kernel", DECODE_SOURCES),
                         "peak_source": peak_src}}
    del S, snap, conv_in, conv_out, tq, tz, tg, tb, od

    # the projections around the mixer at the 27B shape, 8192 tokens
    Tp = 8192
    for name, K, N, split in (("in_proj", 5120, 16480, True), ("out_proj", 6144, 5120, False)):
        xa, wa = I.linear_problem(Tp, N, K, case=rank_case(80 + (name == "out_proj"), rank))
        x_, w_ = dev(xa, bf), dev(wa, bf)
        if split:  # straight into the mixer's input buffers: qkv_pre | z | b | a
            edges = np.cumsum([0, conv_channels(16, 48), 48 * D, 48, 48])
            outs = [(int(lo), int(hi), torch.empty(Tp, int(hi - lo), device="cuda", dtype=bf))
                    for lo, hi in zip(edges[:-1], edges[1:])]
        else:
            outs = [(0, N, torch.empty(Tp, N, device="cuda", dtype=bf))]
        ms = time_launches(lambda: gdn.gdn_linear(x_, w_, outs, stream=stream), steps, args.warmup,
                           stream, barrier, world)
        fl = 2.0 * Tp * N * K
        tf = fl / (ms * 1e-3) / 1e12
        out["linear_" + name] = {
            "workload": "27B %s: %d tokens, K=%d, N=%d, bf16 in/out, fp32 accumulation%s"
                        % (name, Tp, K, N, ", output split into qkv_pre|z|b|a" if split else ""),
            "value": world * tf, "unit": "TFLOP/s", "ms_per_launch": ms,
            "roofline": {"bound": "tensor", "achieved": tf, "peak": peaks["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": tf / peaks["bf16_tflops"],
                         "peak_source": peak_src + " bf16_tflops (burst)"}}
        del x_, w_, outs
    if gdn.gdn_device_status(stream) != 0:
        raise RuntimeError("device status not OK after the extended calls")
    return out


# --------------------------------------------------------- reference arm
def reference_arm(args, world, rank):
    """The oracle, as it stands, timed on the host cores: rank 0 only."""
    if rank != 0:
        return
    from gated_deltanet_mixer_gb300 import inputs as I
    from oracle import oracle as O

    threads = O.default_threads()
    p = I.case_problem(args.workload)

    # Size one step's sample so that warmup + steps fit in about args.ref_budget seconds.
    per_step = args.ref_budget / max(1, args.steps + args.warmup)
    T_s, _ = oracle_tokens_per_s(p, per_step, threads)

    def step():
        oracle_run(p, T_s, threads)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    secs = (time.perf_counter() - t0) / args.steps
    value = T_s / secs
    sample = ("fp64 oracle on the first %d of the workload's %d tokens per step (%d sequences "
              "x %d), all %d value heads" % (T_s, p.B * p.T, p.B, p.T, p.Hv))
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; model-shaped random inputs, no weights needed)",
        "config": {"workload": workload_name(args.workload, p),
                   "io_dtype": p.io, "state_dtype": "f32"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }))


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["gdn", "reference"], default="gdn")
    ap.add_argument("--workload", default="4b_prefill",
                    choices=["4b_prefill", "0.8b_prefill", "27b_prefill"])
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-shapes", action="store_true",
                    help="skip the other prefill shapes of the metric (0.8B, 27B)")
    ap.add_argument("--no-next", action="store_true",
                    help="skip the extended calls (raw gates, packed batch, multi-token decode)")
    ap.add_argument("--cpu-budget", type=float, default=15.0,
                    help="seconds of oracle work for the cpu_baseline sample")
    ap.add_argument("--ref-budget", type=float, default=120.0,
                    help="seconds of oracle work for the whole reference arm")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")
    world, rank, local = dist_env()
    if args.impl == "reference":
        reference_arm(args, world, rank)
    else:
        gdn_arm(args, world, rank, local)


if __name__ == "__main__":
    main()

"""Benchmark of the Gated DeltaNet speculative/MTP decode step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--graph]

One step = one gdn_spec_decode call (the whole hot path: rewind, gates, q/k
norm, recurrence, slot writes, gated RMSNorm, gather) on one batch of seeded
synthetic inputs already resident in HBM.  Prints ONE JSON line on rank 0.

Workload (default ``bs32_t8_bf16``): BS=32 sequences, H_k=2, H_v=16,
K=V=128, T=8 draft tokens, bf16 state, acceptance U{0..8}, a 4096-slot (2 GiB)
pool.  Eight disjoint slot tables (and eight token-input sets) rotate from
step to step, so the state a step touches (~151 MB) was last touched 7 steps
(~1.2 GB of traffic) earlier: the working set exceeds the 129 MB L2.

Under torchrun (N > 1) each rank runs its own independent batch on its own
GPU (sequences are independent: weak scaling, no collective on the data
path); the timing is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "µs/step and draft-token·head updates/s at BS 4–256; % of GB300 HBM roofline"
UNIT = "draft-token·head updates/s"
N_SETS = 8

WORKLOADS = {
    # name: (description, constructor args)
    "bs32_t8_bf16": ("BS=32, H_k=2, H_v=16, K=V=128, T=8, bf16 state, acceptance U{0..8}, 4096-slot (2 GiB) pool",
                     dict(bs=32, sd="bf16")),
    "bs32_t8_f32": ("BS=32, H_k=2, H_v=16, K=V=128, T=8, fp32 state, acceptance U{0..8}, 2048-slot (2 GiB) pool",
                    dict(bs=32, sd="f32")),
}
for _bs in (4, 8, 16, 64, 128):
    for _sd, _ns in (("bf16", 4096), ("f32", 2048)):
        _slots = max(4 * _bs * 8, _ns, N_SETS * _bs * 8)
        WORKLOADS[f"bs{_bs}_t8_{_sd}"] = (
            f"BS={_bs}, H_k=2, H_v=16, K=V=128, T=8, {_sd} state, acceptance U{{0..8}}, {_slots}-slot pool",
            dict(bs=_bs, sd=_sd))
for _bs, _L in ((4, 1024), (32, 256)):
    WORKLOADS[f"prefill_bs{_bs}_l{_L}_bf16"] = (
        f"prefill: {_bs} prompts x {_L} tokens, H_k=2, H_v=16, K=V=128, bf16 state read from and written to a slot",
        dict(prefill=True, bs=_bs, L=_L))
for _T in (1, 2, 4):     # shallower drafts (the T = 4 point is the BS=32 decode-batch shape)
    WORKLOADS[f"bs32_t{_T}_bf16"] = (
        f"BS=32, H_k=2, H_v=16, K=V=128, T={_T}, bf16 state, acceptance U{{0..{_T}}}, 4096-slot (2 GiB) pool",
        dict(bs=32, sd="bf16", T=_T))
WORKLOADS["bs32_t8_bf16_conv"] = (
    "BS=32, H_k=2, H_v=16, K=V=128, T=8, bf16 state, acceptance U{0..8}, 4096-slot pool, with the width-4 "
    "causal convolution and its rewind fused in front (bf16 conv slots, 2 per sequence per set)",
    dict(bs=32, sd="bf16", conv=True))
WORKLOADS["large_bs256_t8_bf16"] = (
    "BS=256, H_k=4, H_v=32, K=V=128, T=8, bf16 state, acceptance Binomial(8,0.7), 16384-slot (16 GiB) pool",
    dict(large=True))


def make_case(name, seed):
    from gated_deltanet_linear_sm_gb300 import synth
    spec = WORKLOADS[name][1]
    if spec.get("prefill"):
        bs, L = spec["bs"], spec["L"]
        return synth.make_case(batch=bs, H_k=2, H_v=16, T=L, spec_stride=1, q_lens=[L] * bs, acc=[1] * bs,
                               state_dtype=synth.BF16, num_slots=max(2 * N_SETS * bs, 64), seed=seed)
    if spec.get("large"):
        return synth.large(seed, num_slots=N_SETS * 256 * 8)
    sd = {"bf16": synth.BF16, "f32": synth.F32}[spec["sd"]]
    bs, T = spec["bs"], spec.get("T", 8)
    ns = max(synth.sweep_num_slots(bs, T, sd), N_SETS * bs * T)
    return synth.sweep(bs, sd, T=T, seed=seed, num_slots=ns)


# ---------------------------------------------------------------------------
# clocks during the timed region (nvidia-smi, read only)
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}", "--format=csv,noheader",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, which):
        if which == "start":
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        for t, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm = float(parts[1].split()[0])
                smax = float(parts[2].split()[0])
            except ValueError:
                continue
            reasons = []
            for name, val in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"),
                                 parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.append(name)
            rows.append((t, sm, smax, reasons))
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        inside = [r for r in rows if self.t0 is not None and self.t0 - 0.06 <= r[0] <= (self.t1 or 1e18) + 0.06]
        use = inside if inside else [r for r in rows if self.t0 is not None and abs(r[0] - self.t0) < 0.5] or rows
        reasons = sorted({x for r in use for x in r[3]})
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
                "reasons": reasons, "samples": len(use), "samples_in_region": len(inside)}


# ---------------------------------------------------------------------------
# roofline helpers
# ---------------------------------------------------------------------------

def measured_peak_gbs():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


KERNEL_SOURCES = ("gated_deltanet_linear_sm_gb300/csrc/gdnspec.cu",
                  "gated_deltanet_linear_sm_gb300/csrc/gdnprefill_chunked.cu",
                  "gated_deltanet_linear_sm_gb300/csrc/gdn_internal.h")


def kernel_source_hash():
    """First 16 hex digits of the SHA-256 of the kernel sources."""
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload):
    """DRAM bytes per launch from the committed ncu summary for this workload
    (profiles/<kernel>_<workload>.md), if it was taken on the current kernel
    sources; else None."""
    import glob
    paths = sorted(glob.glob(os.path.join(ROOT, "profiles", f"*_{workload}.md")))
    try:
        text = open(paths[0]).read()
    except (OSError, IndexError):
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*(\d+)", text)
    s = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    if not m or not s or s.group(1) != kernel_source_hash():
        return None
    return int(m.group(1))



# ---------------------------------------------------------------------------
# the CUDA runtime through ctypes, for the end-to-end leg's copies and events
# ---------------------------------------------------------------------------

class CudaRuntime:
    H2D, D2H = 1, 2

    def __init__(self):
        import ctypes
        import glob
        cands = []
        for d in (os.environ.get("CUDA_HOME", "/usr/local/cuda"), "/usr/local/cuda"):
            cands += sorted(glob.glob(os.path.join(d, "lib64", "libcudart.so*")))
        lib = None
        for c in cands + ["libcudart.so"]:
            try:
                lib = ctypes.CDLL(c)
                break
            except OSError:
                continue
        if lib is None:
            raise RuntimeError("libcudart not found")
        vp, sz = ctypes.c_void_p, ctypes.c_size_t
        lib.cudaMemcpyAsync.argtypes = [vp, vp, sz, ctypes.c_int, vp]
        lib.cudaEventCreateWithFlags.argtypes = [ctypes.POINTER(vp), ctypes.c_uint]
        lib.cudaEventRecord.argtypes = [vp, vp]
        lib.cudaStreamWaitEvent.argtypes = [vp, vp, ctypes.c_uint]
        self.lib, self.ctypes = lib, ctypes

    def _ok(self, rc, what):
        if rc != 0:
            raise RuntimeError(f"{what} failed: {rc}")

    def event(self):
        ev = self.ctypes.c_void_p()
        self._ok(self.lib.cudaEventCreateWithFlags(self.ctypes.byref(ev), 2), "cudaEventCreateWithFlags")
        return ev

    def copy(self, dst, src, n, kind, stream):
        self._ok(self.lib.cudaMemcpyAsync(dst, src, n, kind, stream), "cudaMemcpyAsync")

    def record(self, ev, stream):
        self._ok(self.lib.cudaEventRecord(ev, stream), "cudaEventRecord")

    def wait(self, stream, ev):
        self._ok(self.lib.cudaStreamWaitEvent(stream, ev, 0), "cudaStreamWaitEvent")


# ---------------------------------------------------------------------------
# multi-rank helpers (independent batches per rank; no data-path collective)
# ---------------------------------------------------------------------------

def max_over_ranks(x, world, device):
    """The slowest rank's time: every rank gets max(x) over the group."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(updates_per_rank, world, elapsed_ms_max, steps):
    """Updates all ranks processed per second of the slowest rank's time."""
    return updates_per_rank * world / (elapsed_ms_max * 1e-3 / steps)


def rank_seed(rank):
    """Each rank draws its own independent batch."""
    return rank

# ---------------------------------------------------------------------------
# CPU arm: the oracle, timed as it stands, on the host cores
# ---------------------------------------------------------------------------

def time_oracle(case, seqs=None, min_wall=1.5, max_steps=None):
    """Run the oracle on the given sequences of the workload (default: all)
    repeatedly until min_wall seconds or max_steps runs; returns throughput."""
    from gated_deltanet_linear_sm_gb300 import synth
    from oracle import oracle as orc

    threads = os.cpu_count() or 1
    seqs = list(range(case.batch)) if seqs is None else list(seqs)
    sub, slot_map, _ = synth.subset(case, seqs)
    bits = case.slot_values(slot_map)
    updates = synth.token_head_updates(sub)
    steps = 0
    wall = 0.0
    while True:
        pool = np.ascontiguousarray(bits.copy())
        t0 = time.perf_counter()
        orc.run_case(sub, pool, num_threads=threads)
        wall += time.perf_counter() - t0
        steps += 1
        if (steps >= max_steps) if max_steps else (wall >= min_wall):
            break
    return {"value": updates * steps / wall, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{steps} run(s) of {len(seqs)} of the workload's {case.batch} sequences x "
                      f"{case.H_v} v-heads x up to 8 tokens; FP64 scalar C, OpenMP over "
                      f"(sequence, v-head); {wall:.2f} s wall",
            "seconds": wall, "steps": steps}


def run_reference(args, rank, world):
    """--impl reference: the oracle as the reference arm, rank 0 only."""
    if rank != 0:
        return
    case = make_case(args.workload, seed=0)
    # one step = the oracle on one sequence of the workload (all its v-heads
    # and draft tokens), a bounded sample so that K steps finish in seconds
    for _ in range(args.warmup):
        time_oracle(case, seqs=[0], min_wall=0.0, max_steps=1)
    r = time_oracle(case, seqs=[0], min_wall=0.0, max_steps=args.steps)
    ms = r["seconds"] / r["steps"] * 1e3
    line = {
        "impl": "reference", "metric": METRIC, "value": r["value"], "unit": UNIT, "n_gpus": 0,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{args.workload}: {WORKLOADS[args.workload][0]}", "global_batch": case.batch,
                   "seq_len": 8, "parallelism": "host cores"},
        "cpu_baseline": {"value": r["value"], "unit": UNIT, "cores": r["cores"], "kind": "oracle",
                         "sample": r["sample"]},
        "e2e": {"value": r["value"], "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def run_ours(args, rank, world, local_rank):
    import torch

    import gated_deltanet_linear_sm_gb300 as gdn
    from gated_deltanet_linear_sm_gb300 import synth

    gdn.load_library()                      # fail loudly if the library is missing
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    case = make_case(args.workload, seed=rank_seed(rank))
    sets = synth.disjoint_index_sets(case, N_SETS)
    tdt = {synth.F32: torch.float32, synth.BF16: torch.bfloat16, synth.F16: torch.float16}[case.state_dtype]

    def bf(x):
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to(dev).view(torch.bfloat16)

    # --- resident inputs: the pool and N_SETS token-input / slot-table sets ---
    g = torch.Generator(device=dev)
    g.manual_seed(1000 + rank)
    pool = torch.randn((case.num_slots, case.H_v, case.K, case.V), generator=g, device=dev, dtype=torch.float32)
    pool = pool.mul_(0.1).to(tdt)
    # Each set's per-step inputs live in one contiguous device buffer (views
    # carved at 256-byte boundaries), so the end-to-end leg moves a step's
    # inputs with a single host-to-device copy.
    fields = [("q", torch.bfloat16, case.q.shape), ("k", torch.bfloat16, case.k.shape),
              ("v", torch.bfloat16, case.v.shape), ("a", torch.bfloat16, case.a.shape),
              ("b", torch.bfloat16, case.b.shape), ("z", torch.bfloat16, case.z.shape),
              ("state_indices", torch.int32, case.state_indices.shape),
              ("num_accepted", torch.int32, case.num_accepted.shape),
              ("cu_seqlens", torch.int32, case.cu_seqlens.shape)]
    offsets, total = {}, 0
    for name, dt, shape in fields:
        offsets[name] = total
        total += (int(np.prod(shape)) * torch.tensor([], dtype=dt).element_size() + 255) // 256 * 256

    def carve(buf):
        views = {}
        for name, dt, shape in fields:
            n = int(np.prod(shape)) * torch.tensor([], dtype=dt).element_size()
            views[name] = buf[offsets[name]:offsets[name] + n].view(dt).view(*shape)
        return views

    def host_bytes(c, slot_table):
        hb = torch.empty(total, dtype=torch.uint8)
        hv = carve(hb)
        for name in ("q", "k", "v", "a", "b", "z"):
            hv[name].copy_(torch.from_numpy(getattr(c, name).view(np.int16)).view(torch.bfloat16))
        hv["state_indices"].copy_(torch.from_numpy(slot_table))
        hv["num_accepted"].copy_(torch.from_numpy(case.num_accepted))
        hv["cu_seqlens"].copy_(torch.from_numpy(case.cu_seqlens))
        return hb

    inputs, host_bufs = [], []
    A_log_d = torch.from_numpy(case.A_log).to(dev)
    dt_bias_d, norm_w_d = bf(case.dt_bias), bf(case.norm_w)
    for s in range(N_SETS):
        c = case if s == 0 else synth.make_case(
            batch=case.batch, H_k=case.H_k, H_v=case.H_v, T=case.spec_stride, state_dtype=case.state_dtype,
            num_slots=case.num_slots, acc=case.num_accepted, seed=100 * rank + s)
        hb = host_bytes(c, sets[s]).pin_memory()
        db = hb.to(dev)
        t = carve(db)
        t.update(buf=db, A_log=A_log_d, dt_bias=dt_bias_d, norm_w=norm_w_d,
                 out=torch.zeros((case.num_tokens, case.H_v, case.V), dtype=torch.bfloat16, device=dev))
        inputs.append(t)
        host_bufs.append((hb, torch.empty_like(t["out"], device="cpu").pin_memory()))
    calls = [gdn.prepare(t["q"], t["k"], t["v"], t["a"], t["b"], t["z"], t["A_log"], t["dt_bias"], t["norm_w"],
                         pool, t["state_indices"], t["num_accepted"], t["cu_seqlens"], t["out"], max_T=8,
                         split=args.split)
             for t in inputs]
    updates = synth.token_head_updates(case)
    alg_bytes = synth.algorithmic_bytes(case)
    stream = torch.cuda.current_stream(dev)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    # --- warm-up ---
    for s in range(max(args.warmup, 3)):
        calls[s % N_SETS](stream)
    torch.cuda.synchronize()

    # --- timed region: exactly K steps, device-timed with CUDA events ---
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except AttributeError:
        gpu_id = str(local_rank)
    sampler = ClockSampler(gpu_id)
    sampler.start()
    # keep the GPU busy while the sampler starts, so the timed region runs at load clocks
    t_soak = time.time()
    n = 0
    while time.time() - t_soak < 0.4:
        calls[n % N_SETS](stream.cuda_stream)
        n += 1
        if n % 64 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    handle = stream.cuda_stream
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler.mark("start")
    t0.record(stream)
    for s in range(args.steps):
        calls[s % N_SETS](handle)
    t1.record(stream)
    torch.cuda.synchronize()
    sampler.mark("end")
    barrier()
    torch.cuda.synchronize()
    elapsed_ms = t0.elapsed_time(t1)
    time.sleep(0.12)
    sampler.stop()
    clocks = sampler.summary()
    elapsed_ms = max_over_ranks(elapsed_ms, world, dev)

    # --- CUDA-graph replay variant: one graph holding one launch per slot set ---
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap):
        for s in range(N_SETS):
            calls[s](cap.cuda_stream)
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    reps = max(args.steps // N_SETS, 1)
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for _ in range(reps):
        graph.replay()
    g1.record(stream)
    torch.cuda.synchronize()
    graph_ms = max_over_ranks(g0.elapsed_time(g1) * args.steps / (reps * N_SETS), world, dev)

    # --- end to end through the public API with host buffers ---
    # every step: one pinned host-to-device copy of the step's inputs, the
    # call, and a device-to-host read of its output.  Copies run on their own
    # streams, so step s+1's inputs travel while step s computes and step s's
    # output travels back while step s+1 computes; events keep each of the
    # N_SETS buffer sets free until the step that last used it has finished.
    h2d = total
    d2h = host_bufs[0][1].numel() * host_bufs[0][1].element_size()
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    rt = CudaRuntime()
    hs, hu, hd = stream.cuda_stream, up.cuda_stream, down.cuda_stream
    h2d_done = [rt.event() for _ in range(N_SETS)]
    run_done = [rt.event() for _ in range(N_SETS)]
    d2h_done = [rt.event() for _ in range(N_SETS)]
    used = [False] * N_SETS
    ptrs = [(hb.data_ptr(), hout.data_ptr(), t["buf"].data_ptr(), t["out"].data_ptr())
            for (hb, hout), t in zip(host_bufs, inputs)]

    def e2e_step(s):
        # plain runtime calls (cudaMemcpyAsync, events) keep the host's share
        # of a step well below the kernel's
        k = s % N_SETS
        h_in, h_out, d_in, d_out = ptrs[k]
        if used[k]:
            rt.wait(hu, run_done[k])                    # the set's inputs were consumed
        rt.copy(d_in, h_in, h2d, rt.H2D, hu)
        rt.record(h2d_done[k], hu)
        rt.wait(hs, h2d_done[k])
        if used[k]:
            rt.wait(hs, d2h_done[k])                    # the set's previous output was read back
        calls[k](hs)
        rt.record(run_done[k], hs)
        rt.wait(hd, run_done[k])
        rt.copy(h_out, d_out, d2h, rt.D2H, hd)
        rt.record(d2h_done[k], hd)
        used[k] = True

    def e2e_drain():
        for k in range(N_SETS):
            if used[k]:
                rt.wait(hs, d2h_done[k])

    for s in range(3):
        e2e_step(s)
    e2e_drain()
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    up.wait_event(e0)
    down.wait_event(e0)
    for s in range(args.steps):
        e2e_step(s)
    e2e_drain()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)

    if rank != 0:
        return
    ms_per_step = elapsed_ms / args.steps
    avg_launch_ms = ms_per_step           # one launch per step, back to back on one stream
    peak, peak_kind = measured_peak_gbs()
    achieved = alg_bytes / (avg_launch_ms * 1e-3) / 1e9
    traffic = profiled_traffic(args.workload)
    cpu = time_oracle(case, seqs=range(min(case.batch, 8)))     # a bounded sample
    line = {
        "metric": METRIC,
        "value": whole_job_value(updates, world, elapsed_ms, args.steps),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "us_per_step": ms_per_step * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {
            "workload": f"{args.workload}: {WORKLOADS[args.workload][0]}",
            "global_batch": case.batch * world,
            "seq_len": 8,
            "parallelism": f"independent batches, {world} GPU(s)",
            "state_dtype": synth.STATE_NAMES[case.state_dtype],
            "cache": "rotating 8 disjoint slot tables and token-input sets; working set > L2",
        },
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_kind": f"{peak_kind} HBM copy bandwidth",
                     "algorithmic_bytes_per_launch": alg_bytes},
        "cpu_baseline": {k: cpu[k] for k in ("value", "unit", "cores", "kind", "sample")},
        "e2e": {"value": whole_job_value(updates, world, e2e_ms, args.steps), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "graph_replay": {"value": whole_job_value(updates, world, graph_ms, args.steps), "unit": UNIT,
                         "us_per_step": graph_ms * 1e3 / args.steps},
        "gpu_launches": args.steps,
        "clocks": clocks,
        "split": gdn.binding.chosen_split(calls[0].dims, calls[0].state_dtype),
    }
    print(json.dumps(line), flush=True)


def run_conv(args, rank, world, local_rank):
    """The fused-conv workload: one step = one gdn_spec_decode_conv call over
    the batch; N_SETS disjoint sets of state-slot tables, conv slot pairs and
    projection rows rotate so that no set is read back from L2."""
    import torch

    import gated_deltanet_linear_sm_gb300 as gdn
    from gated_deltanet_linear_sm_gb300 import synth

    gdn.load_library()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    case = make_case(args.workload, seed=rank_seed(rank))
    B = case.batch
    sets = synth.disjoint_index_sets(case, N_SETS)
    ci = synth.conv_inputs(case, width=4, num_conv_slots=2 * N_SETS * B, seed=rank_seed(rank))

    def bf(x):
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to(dev).view(torch.bfloat16)

    tdt = {synth.F32: torch.float32, synth.BF16: torch.bfloat16, synth.F16: torch.float16}[case.state_dtype]
    g = torch.Generator(device=dev)
    g.manual_seed(1000 + rank)
    pool = torch.randn((case.num_slots, case.H_v, case.K, case.V), generator=g, device=dev).mul_(0.1).to(tdt)
    conv_pool = bf(ci.pool)
    common = dict(A_log=torch.from_numpy(case.A_log).to(dev), dt_bias=bf(case.dt_bias), norm_w=bf(case.norm_w),
                  w=bf(ci.weight), bias=bf(ci.bias), acc=torch.from_numpy(case.num_accepted).to(dev),
                  cu=torch.from_numpy(case.cu_seqlens).to(dev))
    perm = np.random.default_rng(rank).permutation(ci.pool.shape[0]).astype(np.int32)
    per_set = []
    for s in range(N_SETS):
        rng = np.random.default_rng([rank, s, 9])
        x = synth.f32_to_bf16_bits(rng.normal(0, 1, ci.x.shape).astype(np.float32)) if s else ci.x
        per_set.append(dict(
            x=bf(x), a=bf(case.a), b=bf(case.b), z=bf(case.z), idx=torch.from_numpy(sets[s]).to(dev),
            cin=torch.from_numpy(perm[2 * s * B:(2 * s + 1) * B].copy()).to(dev),
            cout=torch.from_numpy(perm[(2 * s + 1) * B:(2 * s + 2) * B].copy()).to(dev)))
    out = torch.zeros((case.num_tokens, case.H_v, case.V), dtype=torch.bfloat16, device=dev)

    def step(s, stream=None):
        d = per_set[s % N_SETS]
        gdn.gdn_spec_decode_conv(d["x"], common["w"], common["bias"], conv_pool, d["cin"], d["cout"], d["a"], d["b"],
                                 d["z"], common["A_log"], common["dt_bias"], common["norm_w"], pool, d["idx"],
                                 common["acc"], common["cu"], out, H_k=case.H_k, max_T=8, stream=stream)

    stream = torch.cuda.current_stream(dev)
    for s in range(max(args.warmup, 3)):
        step(s)
    torch.cuda.synchronize()
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except AttributeError:
        gpu_id = str(local_rank)
    sampler = ClockSampler(gpu_id)
    sampler.start()
    t_soak, n = time.time(), 0
    while time.time() - t_soak < 0.4:                          # load clocks before the timed region
        step(n)
        n += 1
        if n % 64 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler.mark("start")
    e0.record(stream)
    for s in range(args.steps):
        step(s, stream.cuda_stream)
    e1.record(stream)
    torch.cuda.synchronize()
    sampler.mark("end")
    time.sleep(0.12)
    sampler.stop()
    clocks = sampler.summary()
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev) / args.steps
    if rank != 0:
        return
    updates = synth.token_head_updates(case)
    alg = synth.conv_algorithmic_bytes(case, ci)
    peak, peak_kind = measured_peak_gbs()
    achieved = alg / (ms * 1e-3) / 1e9
    print(json.dumps({
        "metric": "token·head updates/s (fused conv + decode)", "value": updates * world / (ms * 1e-3),
        "unit": "token·head updates/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "us_per_step": ms * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"{args.workload}: {WORKLOADS[args.workload][0]}", "global_batch": B * world,
                   "seq_len": 8, "parallelism": f"independent batches, {world} GPU(s)",
                   "l2": f"{N_SETS} rotating input / slot sets"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": profiled_traffic(args.workload), "peak_kind": f"{peak_kind} HBM copy bandwidth",
                     "algorithmic_bytes_per_launch": alg},
        "gpu_launches": args.steps, "clocks": clocks}), flush=True)


def run_prefill(args, rank, world, local_rank):
    """Prefill workloads: one step = one gdn_prefill call over the batch of
    prompts; each prompt starts from a slot and stores its final state in
    another, rotating over N_SETS disjoint slot pairs."""
    import torch

    import gated_deltanet_linear_sm_gb300 as gdn
    from gated_deltanet_linear_sm_gb300 import synth

    gdn.load_library()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    case = make_case(args.workload, seed=rank_seed(rank))
    B = case.batch

    def bf(x):
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to(dev).view(torch.bfloat16)

    pool = (torch.randn((case.num_slots, case.H_v, case.K, case.V), device=dev) * 0.1).to(torch.bfloat16)
    t = dict(q=bf(case.q), k=bf(case.k), v=bf(case.v), a=bf(case.a), b=bf(case.b), z=bf(case.z),
             A_log=torch.from_numpy(case.A_log).to(dev), dt_bias=bf(case.dt_bias), norm_w=bf(case.norm_w),
             cu=torch.from_numpy(case.cu_seqlens).to(dev),
             out=torch.zeros((case.num_tokens, case.H_v, case.V), dtype=torch.bfloat16, device=dev))
    perm = np.random.default_rng(rank).permutation(case.num_slots).astype(np.int32)
    pairs = [(torch.from_numpy(perm[2 * s * B:(2 * s + 1) * B].copy()).to(dev),
              torch.from_numpy(perm[(2 * s + 1) * B:(2 * s + 2) * B].copy()).to(dev)) for s in range(N_SETS)]

    fn = gdn.gdn_prefill_chunked if args.prefill_form == "chunked" else gdn.gdn_prefill

    def step(s, stream=None):
        rd, wr = pairs[s % N_SETS]
        fn(t["q"], t["k"], t["v"], t["a"], t["b"], t["z"], t["A_log"], t["dt_bias"], t["norm_w"],
           pool, rd, wr, t["cu"], t["out"], stream=stream)

    stream = torch.cuda.current_stream(dev)
    for s in range(max(args.warmup, 3)):
        step(s)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for s in range(args.steps):
        step(s, stream.cuda_stream)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev) / args.steps
    if rank != 0:
        return
    tokens = int(case.cu_seqlens[-1])
    updates = tokens * case.H_v
    state_bytes = B * case.H_v * case.K * case.V * 2 * 2            # one tile read, one written
    token_bytes = tokens * (case.H_k * 2 * case.K * 2 + case.H_v * (3 * case.V * 2 + 4))
    alg = state_bytes + token_bytes
    peak, peak_kind = measured_peak_gbs()
    achieved = alg / (ms * 1e-3) / 1e9
    print(json.dumps({
        "metric": "prefill token·head updates/s", "value": updates * world / (ms * 1e-3),
        "unit": "token·head updates/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": f"{args.workload}: {WORKLOADS[args.workload][0]}", "form": args.prefill_form,
                   "global_batch": B * world,
                   "seq_len": int(case.q_lens().max()), "parallelism": f"independent batches, {world} GPU(s)"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": profiled_traffic(args.workload) if args.prefill_form == "chunked" else None,
                     "peak_kind": f"{peak_kind} HBM copy bandwidth", "algorithmic_bytes_per_launch": alg},
        "gpu_launches": args.steps}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="bs32_t8_bf16")
    ap.add_argument("--split", type=lambda x: int(x, 0), default=0,
                    help="decode workloads: dims.split (0 = the library's choice; 1, 2, 4, 8, 0x102, 0x104)")
    ap.add_argument("--prefill-form", choices=("chunked", "recurrent"), default="chunked",
                    help="prefill workloads: gdn_prefill_chunked (tensor cores) or gdn_prefill (per token)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    try:
        if WORKLOADS[args.workload][1].get("prefill"):
            run_prefill(args, rank, world, local_rank)
        elif WORKLOADS[args.workload][1].get("conv"):
            run_conv(args, rank, world, local_rank)
        else:
            run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()

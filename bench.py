"""Benchmark of the Gated DeltaNet speculative/MTP decode step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--split S] [--flags F] [--prefill-form chunked|recurrent]

One step = one library call over one batch of seeded synthetic inputs that are
already resident in HBM: for the decode workloads one gdn_spec_decode call
(the whole hot path: rewind, gates, q/k norm, recurrence, slot writes, gated
RMSNorm, gather).  Prints ONE JSON line on rank 0.

Default workload ``bs32_t8_bf16``: BS=32 sequences, H_k=2, H_v=16, K=V=128,
T=8 draft tokens, bf16 state, acceptance U{0..8}, a 4096-slot (2 GiB) pool.

Cold cache.  Every workload rotates over n_sets input sets (token rows, index
tables and disjoint state slots), n_sets chosen so that the bytes a step
touches were last touched at least twice the L2 size of traffic earlier
(at least 8 sets).  Besides the back-to-back throughput the line reports the
per-step time over 64 windows of one rotation each (median, p10, p90) and 64
single calls each preceded by a 512 MiB scratch write (median, p10, p90).

Under torchrun (N > 1) each rank runs its own independent batch on its own
GPU (sequences are independent: weak scaling, no collective on the data
path); the timing is the max over ranks.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
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
L2_BYTES = 129 * 10 ** 6          # GB300 L2
MIN_SETS = 8
FLUSH_BYTES = 512 << 20
N_WINDOWS = 64
N_COLD = 64

GDN_PRE_INDEX, GDN_PRE_TOKENS, GDN_PRE_STATE = 0x1, 0x2, 0x4

# name: (description, spec)
WORKLOADS = {
    "bs32_t8_bf16": ("BS=32, H_k=2, H_v=16, K=V=128, T=8, bf16 state, acceptance U{0..8}, 4096-slot (2 GiB) pool",
                     dict(bs=32, sd="bf16")),
    "bs32_t8_f32": ("BS=32, H_k=2, H_v=16, K=V=128, T=8, fp32 state, acceptance U{0..8}, 2048-slot (2 GiB) pool",
                    dict(bs=32, sd="f32")),
    "bs32_t8_f16": ("BS=32, H_k=2, H_v=16, K=V=128, T=8, fp16 state, acceptance U{0..8}, 4096-slot (2 GiB) pool",
                    dict(bs=32, sd="f16")),
    "mixed_c3_f16": ("mixed batch: 48 spec sequences (T=3) among 80 non-spec rows (224 token rows), H_k=2, "
                     "H_v=16, K=V=128, q/k/v/a/b/z gathered through spec_token_indx, 10% of slot entries -1, "
                     "acceptance U{0..3}, fp16 state, 4096-slot (2 GiB) pool", dict(mixed=True)),
}
for _bs in (4, 8, 16, 64, 128):
    for _sd in ("bf16", "f32"):
        _slots = 4096 if _sd == "bf16" else 2048
        WORKLOADS[f"bs{_bs}_t8_{_sd}"] = (
            f"BS={_bs}, H_k=2, H_v=16, K=V=128, T=8, {_sd} state, acceptance U{{0..8}}, "
            f">= {_slots}-slot (2 GiB) pool", dict(bs=_bs, sd=_sd))
for _T in (1, 2, 4):     # shallower drafts (the T = 4 point is the BS=32 decode-batch shape)
    WORKLOADS[f"bs32_t{_T}_bf16"] = (
        f"BS=32, H_k=2, H_v=16, K=V=128, T={_T}, bf16 state, acceptance U{{0..{_T}}}, 4096-slot (2 GiB) pool",
        dict(bs=32, sd="bf16", T=_T))
WORKLOADS["large_bs256_t8_bf16"] = (
    "BS=256, H_k=4, H_v=32, K=V=128, T=8, bf16 state, acceptance Binomial(8,0.7), 16384-slot (16 GiB) pool",
    dict(large=True))
WORKLOADS["bs32_t8_bf16_conv"] = (
    "BS=32, H_k=2, H_v=16, K=V=128, T=8, bf16 state, acceptance U{0..8}, 4096-slot pool, with the width-4 "
    "causal convolution and its rewind fused in front (bf16 conv slots, 2 per sequence per set)",
    dict(bs=32, sd="bf16", conv=True))
for _bs, _L in ((4, 1024), (32, 256)):
    WORKLOADS[f"prefill_bs{_bs}_l{_L}_bf16"] = (
        f"prefill: {_bs} prompts x {_L} tokens, H_k=2, H_v=16, K=V=128, bf16 state read from one slot and "
        f"written to another", dict(prefill=True, bs=_bs, L=_L))


def kind_of(name):
    spec = WORKLOADS[name][1]
    return "prefill" if spec.get("prefill") else "conv" if spec.get("conv") else "decode"


def make_case(name, seed, num_slots=None):
    """The workload's synthetic batch for one input set (a synth.Case)."""
    from gated_deltanet_linear_sm_gb300 import synth
    spec = WORKLOADS[name][1]
    if spec.get("prefill"):
        bs, L = spec["bs"], spec["L"]
        return synth.make_case(batch=bs, H_k=2, H_v=16, T=L, spec_stride=1, q_lens=[L] * bs, acc=[1] * bs,
                               state_dtype=synth.BF16, num_slots=num_slots or 2 * MIN_SETS * bs, seed=seed)
    if spec.get("large"):
        return synth.large(seed, num_slots=num_slots or 16384)
    if spec.get("mixed"):
        c = synth.mixed(seed)
        ns = num_slots or synth.sweep_num_slots(48, 3, synth.F16)
        return dataclasses.replace(c, num_slots=ns)
    sd = {"bf16": synth.BF16, "f32": synth.F32, "f16": synth.F16}[spec["sd"]]
    bs, T = spec["bs"], spec.get("T", 8)
    ns = num_slots or synth.sweep_num_slots(bs, T, sd)
    return synth.sweep(bs, sd, T=T, seed=seed, num_slots=ns)


def draft_depth(name):
    spec = WORKLOADS[name][1]
    if spec.get("prefill"):
        return spec["L"]
    if spec.get("mixed"):
        return 3
    return spec.get("T", 8)


def metric_unit(name):
    """The line's metric and unit for a workload."""
    kind = kind_of(name)
    if kind == "prefill":
        return "prefill token·head updates/s", "token·head updates/s"
    if kind == "conv":
        return "token·head updates/s (fused conv + decode)", "token·head updates/s"
    return METRIC, UNIT


def n_sets_for(step_bytes):
    """Input sets to rotate over so that a step's bytes were last touched at
    least 2 x L2 of traffic earlier."""
    return max(MIN_SETS, math.ceil(2 * L2_BYTES / max(step_bytes, 1)) + 1)


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

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, "fallback"


def measured_peak_gbs():
    hbm, _, kind = measured_peaks()
    return hbm, kind


CSRC = "gated_deltanet_linear_sm_gb300/csrc/"
# the sources of the kernel each kind of workload times
KERNEL_SOURCES = {"decode": (CSRC + "gdnspec.cu", CSRC + "gdn_internal.h"),
                  "conv": (CSRC + "gdnspec.cu", CSRC + "gdn_internal.h"),
                  "prefill": (CSRC + "gdnprefill_chunked.cu", CSRC + "gdn_internal.h")}


def kernel_source_hash(kind="decode"):
    """First 16 hex digits of the SHA-256 of the timed kernel's sources."""
    h = hashlib.sha256()
    for p in KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload):
    """DRAM bytes per launch from the committed ncu summary for this workload
    (profiles/<kernel>_<workload>.md), if it was taken on the current sources
    of the timed kernel; else None."""
    import glob
    paths = sorted(glob.glob(os.path.join(ROOT, "profiles", f"*_{workload}.md")))
    try:
        text = open(paths[0]).read()
    except (OSError, IndexError):
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*(\d+)", text)
    s = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    if not m or not s or s.group(1) != kernel_source_hash(kind_of(workload)):
        return None
    return int(m.group(1))


def prefill_alg_bytes(case):
    """Bytes a prefill call must move: one state tile read and one written per
    (prompt, v-head), and every token row (q, k per k-head; v, z, out, a, b
    per v-head)."""
    tokens = int(case.cu_seqlens[-1])
    return (case.batch * case.H_v * case.K * case.V * 2 * 2
            + tokens * (case.H_k * 2 * case.K * 2 + case.H_v * (3 * case.V * 2 + 4)))


def chunked_prefill_flops(case, chunk=64):
    """FLOPs of the chunked form's products per launch (two per multiply-add),
    per (prompt, v-head) and chunk of n tokens: K^ K^^T and Q^ K^^T (n x n x
    K each), K^ S and Q^ S (n x V x K each), R~ V' (n x n x V) and the state
    update K~^T V' (K x V x n)."""
    K, V = case.K, case.V
    total = 0
    for L in case.q_lens():
        for c0 in range(0, int(L), chunk):
            n = min(chunk, int(L) - c0)
            total += 2 * (2 * n * n * K + 2 * n * V * K + n * n * V + K * V * n)
    return total * case.H_v


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


def pct(xs, q):
    return float(np.percentile(np.asarray(xs, dtype=np.float64), q))


# ---------------------------------------------------------------------------
# CPU side: the oracle, timed as it stands, on the host cores
# ---------------------------------------------------------------------------

def _oracle_runner(name, case):
    """(fn(threads) running the oracle once on a bounded sample of `case`,
    token·head updates of one run, description of the sample)."""
    from gated_deltanet_linear_sm_gb300 import synth
    from oracle import oracle as orc
    kind = kind_of(name)
    if kind == "prefill":
        sub, _, _ = synth.subset(case, [0])          # one prompt, all its v-heads and tokens
        rd = np.array([0], np.int32)
        wr = np.array([1], np.int32)
        bits = case.slot_values([0, 1])
        updates = int(sub.q_lens().sum()) * sub.H_v

        def fn(threads):
            pool = np.ascontiguousarray(bits.copy())
            orc.prefill(q=sub.q, k=sub.k, v=sub.v, a=sub.a, b=sub.b, z=sub.z, A_log=sub.A_log,
                        dt_bias=sub.dt_bias, norm_w=sub.norm_w, pool=pool, state_dtype=sub.state_dtype,
                        cu_seqlens=sub.cu_seqlens, read_slots=rd, write_slots=wr, num_threads=threads)
        return fn, updates, f"1 of the workload's {case.batch} prompts ({int(sub.q_lens().sum())} tokens) x " \
                            f"{case.H_v} v-heads"
    seqs = list(range(min(case.batch, 8)))
    sub, slot_map, _ = synth.subset(case, seqs)
    bits = case.slot_values(slot_map)
    updates = synth.token_head_updates(sub)
    desc = f"{len(seqs)} of the workload's {case.batch} sequences x {case.H_v} v-heads x up to " \
           f"{draft_depth(name)} tokens"
    if kind == "decode":
        def fn(threads):
            orc.run_case(sub, np.ascontiguousarray(bits.copy()), num_threads=threads)
        return fn, updates, desc
    ci = synth.conv_inputs(sub, width=4, seed=0)

    def fn(threads):
        orc.spec_decode_conv(x=ci.x, conv_weight=ci.weight, conv_bias=ci.bias, conv_pool=ci.pool.copy(),
                             conv_in=ci.conv_in, conv_out=ci.conv_out, H_k=sub.H_k, K=sub.K, a=sub.a, b=sub.b,
                             z=sub.z, A_log=sub.A_log, dt_bias=sub.dt_bias, norm_w=sub.norm_w,
                             pool=np.ascontiguousarray(bits.copy()), state_dtype=sub.state_dtype,
                             state_indices=sub.state_indices, num_accepted=sub.num_accepted,
                             cu_seqlens=sub.cu_seqlens, num_threads=threads)
    return fn, updates, desc + ", with the width-4 convolution"


def time_oracle(name, case, min_wall=1.5, max_steps=None, threads=None):
    """Run the oracle on a bounded sample of the workload repeatedly until
    min_wall seconds or max_steps runs; returns its throughput."""
    threads = threads or os.cpu_count() or 1
    fn, updates, desc = _oracle_runner(name, case)
    steps, wall = 0, 0.0
    while True:
        t0 = time.perf_counter()
        fn(threads)
        wall += time.perf_counter() - t0
        steps += 1
        if (steps >= max_steps) if max_steps else (wall >= min_wall):
            break
    return {"value": updates * steps / wall, "unit": metric_unit(name)[1], "cores": threads, "kind": "oracle",
            "sample": f"{steps} run(s) of {desc}; FP64 scalar C, OpenMP over (sequence, v-head) on "
                      f"{threads} thread(s); {wall:.2f} s wall",
            "seconds": wall, "steps": steps}


def cpu_baseline(name, case):
    """The oracle on all host cores and on one, each for ~1.5 s wall."""
    multi = time_oracle(name, case)
    single = time_oracle(name, case, threads=1)
    d = {k: multi[k] for k in ("value", "unit", "cores", "kind", "sample")}
    d["single_thread"] = {"value": single["value"], "sample": single["sample"]}
    return d


def run_reference(args, rank, world):
    """--impl reference: the oracle as the reference arm, rank 0 only."""
    if rank != 0:
        return
    case = make_case(args.workload, seed=0)
    # one step = the oracle on a bounded sample of the workload (see
    # _oracle_runner), so that K steps finish in seconds
    for _ in range(args.warmup):
        time_oracle(args.workload, case, min_wall=0.0, max_steps=1)
    r = time_oracle(args.workload, case, min_wall=0.0, max_steps=args.steps)
    ms = r["seconds"] / r["steps"] * 1e3
    metric, unit = metric_unit(args.workload)
    line = {
        "impl": "reference", "metric": metric, "value": r["value"], "unit": unit, "n_gpus": 0,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{args.workload}: {WORKLOADS[args.workload][0]}", "global_batch": case.batch,
                   "seq_len": draft_depth(args.workload), "parallelism": "host cores"},
        "cpu_baseline": {"value": r["value"], "unit": unit, "cores": r["cores"], "kind": "oracle",
                         "sample": r["sample"]},
        "e2e": {"value": r["value"], "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# GPU side: rotating input sets
# ---------------------------------------------------------------------------

class Packed:
    """The per-step inputs of one set in one contiguous device buffer (views
    carved at 256-byte boundaries) with a pinned host copy of the same
    layout, so that the end-to-end leg moves a step's inputs in one copy."""

    def __init__(self, dev, fields):
        import torch
        self.offsets, total = {}, 0
        for name, arr in fields:
            self.offsets[name] = total
            total += (arr.nbytes + 255) // 256 * 256
        self.total = total
        self.host = torch.zeros(total, dtype=torch.uint8).pin_memory()
        hv = self.host.numpy()
        for name, arr in fields:
            o = self.offsets[name]
            hv[o:o + arr.nbytes] = np.ascontiguousarray(arr).view(np.uint8).ravel()
        self.dev = self.host.to(dev)
        self.views = {}
        for name, arr in fields:
            o = self.offsets[name]
            raw = self.dev[o:o + arr.nbytes]
            if arr.dtype == np.uint16:          # bf16 bits
                t = raw.view(torch.int16).view(torch.bfloat16)
            elif arr.dtype == np.int32:
                t = raw.view(torch.int32)
            else:
                t = raw.view(torch.float32)
            self.views[name] = t.view(*arr.shape)


@dataclasses.dataclass
class StepSet:
    call: object                # call(handle, flags) launches one step on the stream handle
    packed: Packed
    out: object                 # device output tensor
    host_out: object            # pinned host tensor of the same size
    updates: int
    alg_bytes: int
    flops: int = 0
    prepared: object = None     # decode: the marshalled call (for its dims)


def disjoint_slot_tables(cases, num_slots, rng):
    """One slot table per set, pairwise disjoint, each keeping its case's -1
    pattern."""
    need = sum(c.state_indices.size for c in cases)
    if need > num_slots:
        raise ValueError(f"{len(cases)} disjoint sets need {need} slots > {num_slots}")
    perm = rng.permutation(num_slots).astype(np.int32)
    out, o = [], 0
    for c in cases:
        n = c.state_indices.size
        t = perm[o:o + n].reshape(c.state_indices.shape).copy()
        t[c.state_indices < 0] = -1
        out.append(t)
        o += n
    return out


def build_sets(args, rank, dev):
    """The workload's rotating input sets on the device, its state pool and
    the first set's case (for the oracle leg)."""
    import torch

    import gated_deltanet_linear_sm_gb300 as gdn
    from gated_deltanet_linear_sm_gb300 import synth

    name = args.workload
    kind = kind_of(name)
    case0 = make_case(name, seed=1000 * rank)
    step_bytes = prefill_alg_bytes(case0) if kind == "prefill" else synth.algorithmic_bytes(case0)
    n_sets = n_sets_for(step_bytes)
    per_set_slots = case0.state_indices.size if kind != "prefill" else 2 * case0.batch
    num_slots = max(case0.num_slots, n_sets * per_set_slots)
    cases = [make_case(name, seed=1000 * rank + s, num_slots=num_slots) for s in range(n_sets)]
    tdt = {synth.F32: torch.float32, synth.BF16: torch.bfloat16, synth.F16: torch.float16}[case0.state_dtype]
    g = torch.Generator(device=dev)
    g.manual_seed(1000 + rank)
    pool = torch.empty((num_slots, case0.H_v, case0.K, case0.V), dtype=tdt, device=dev)
    for s0 in range(0, num_slots, 256):          # N(0, 0.1) in slabs (no full-size FP32 temporary)
        s1 = min(num_slots, s0 + 256)
        pool[s0:s1] = (torch.randn((s1 - s0,) + tuple(pool.shape[1:]), generator=g, device=dev) * 0.1).to(tdt)

    def bf(x):
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to(dev).view(torch.bfloat16)

    A_log = torch.from_numpy(case0.A_log).to(dev)
    dt_bias, norm_w = bf(case0.dt_bias), bf(case0.norm_w)
    rng = np.random.default_rng([rank, 7])
    sets = []
    if kind == "prefill":
        perm = rng.permutation(num_slots).astype(np.int32)
        fn = gdn.gdn_prefill_chunked if args.prefill_form == "chunked" else gdn.gdn_prefill
        for s, c in enumerate(cases):
            B = c.batch
            pk = Packed(dev, [("q", c.q), ("k", c.k), ("v", c.v), ("a", c.a), ("b", c.b), ("z", c.z),
                              ("read", perm[2 * s * B:(2 * s + 1) * B]),
                              ("write", perm[(2 * s + 1) * B:(2 * s + 2) * B]), ("cu", c.cu_seqlens)])
            v = pk.views
            out = torch.zeros((c.num_tokens, c.H_v, c.V), dtype=torch.bfloat16, device=dev)

            def call(handle, flags, v=v, out=out):
                fn(v["q"], v["k"], v["v"], v["a"], v["b"], v["z"], A_log, dt_bias, norm_w, pool, v["read"],
                   v["write"], v["cu"], out, stream=handle)
            sets.append(StepSet(call, pk, out, torch.empty_like(out, device="cpu").pin_memory(),
                                int(c.cu_seqlens[-1]) * c.H_v, prefill_alg_bytes(c), chunked_prefill_flops(c)))
        return sets, pool, cases[0], n_sets, num_slots
    tables = disjoint_slot_tables(cases, num_slots, rng)
    if kind == "conv":
        D = 2 * case0.H_k * case0.K + case0.H_v * case0.V
        ci0 = synth.conv_inputs(case0, width=4, num_conv_slots=2 * n_sets * case0.batch, seed=rank)
        conv_pool, conv_w, conv_b = bf(ci0.pool), bf(ci0.weight), bf(ci0.bias)
        cperm = rng.permutation(ci0.pool.shape[0]).astype(np.int32)
        for s, c in enumerate(cases):
            B = c.batch
            x = ci0.x if s == 0 else synth.f32_to_bf16_bits(
                np.random.default_rng([rank, s, 9]).normal(0, 1, (c.num_tokens, D)).astype(np.float32))
            pk = Packed(dev, [("x", x), ("a", c.a), ("b", c.b), ("z", c.z), ("idx", tables[s]),
                              ("acc", c.num_accepted), ("cu", c.cu_seqlens),
                              ("cin", cperm[2 * s * B:(2 * s + 1) * B]),
                              ("cout", cperm[(2 * s + 1) * B:(2 * s + 2) * B])])
            v = pk.views
            out = torch.zeros((c.num_tokens, c.H_v, c.V), dtype=torch.bfloat16, device=dev)

            def call(handle, flags, v=v, out=out, c=c):
                gdn.gdn_spec_decode_conv(v["x"], conv_w, conv_b, conv_pool, v["cin"], v["cout"], v["a"], v["b"],
                                         v["z"], A_log, dt_bias, norm_w, pool, v["idx"], v["acc"], v["cu"], out,
                                         H_k=c.H_k, max_T=8, flags=flags, stream=handle)
            cs = dataclasses.replace(c, state_indices=tables[s])
            ci = dataclasses.replace(ci0, x=x, conv_in=cperm[2 * s * B:(2 * s + 1) * B],
                                     conv_out=cperm[(2 * s + 1) * B:(2 * s + 2) * B])
            sets.append(StepSet(call, pk, out, torch.empty_like(out, device="cpu").pin_memory(),
                                synth.token_head_updates(cs), synth.conv_algorithmic_bytes(cs, ci)))
        return sets, pool, cases[0], n_sets, num_slots
    for s, c in enumerate(cases):
        fields = [("q", c.q), ("k", c.k), ("v", c.v), ("a", c.a), ("b", c.b), ("z", c.z), ("idx", tables[s]),
                  ("acc", c.num_accepted), ("cu", c.cu_seqlens)]
        if c.spec_token_indx is not None:
            fields.append(("sti", c.spec_token_indx))
        pk = Packed(dev, fields)
        v = pk.views
        out = torch.zeros((c.num_tokens, c.H_v, c.V), dtype=torch.bfloat16, device=dev)
        calls = {}
        for flags in {args.flags, 0}:
            calls[flags] = gdn.prepare(v["q"], v["k"], v["v"], v["a"], v["b"], v["z"], A_log, dt_bias, norm_w,
                                       pool, v["idx"], v["acc"], v["cu"], out, spec_token_indx=v.get("sti"),
                                       max_T=8, split=args.split, flags=flags)

        def call(handle, flags, calls=calls):
            calls[flags](handle)
        cs = dataclasses.replace(c, state_indices=tables[s])
        sets.append(StepSet(call, pk, out, torch.empty_like(out, device="cpu").pin_memory(),
                            synth.token_head_updates(cs), synth.algorithmic_bytes(cs), prepared=calls[args.flags]))
    return sets, pool, cases[0], n_sets, num_slots


def run_gpu(args, rank, world, local_rank):
    import torch

    import gated_deltanet_linear_sm_gb300 as gdn
    from gated_deltanet_linear_sm_gb300 import synth

    gdn.load_library()                      # fail loudly if the library is missing
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    name = args.workload
    kind = kind_of(name)
    flags = args.flags if kind != "prefill" else 0
    sets, pool, case0, n_sets, num_slots = build_sets(args, rank, dev)
    stream = torch.cuda.current_stream(dev)
    handle = stream.cuda_stream
    K = args.steps

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    def steps(n, fl=flags, h=handle, start=0):
        for s in range(start, start + n):
            sets[s % n_sets].call(h, fl)

    updates_k = sum(sets[s % n_sets].updates for s in range(K))
    bytes_k = sum(sets[s % n_sets].alg_bytes for s in range(K))
    flops_k = sum(sets[s % n_sets].flops for s in range(K))

    # --- warm-up ---
    steps(max(args.warmup, 3))
    torch.cuda.synchronize()

    # --- timed region: exactly K steps back to back, device-timed with CUDA events ---
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except AttributeError:
        gpu_id = str(local_rank)
    sampler = ClockSampler(gpu_id)
    sampler.start()
    t_soak, n = time.time(), 0               # load clocks before the timed region
    while time.time() - t_soak < 0.4:
        steps(n_sets, start=n)
        n += n_sets
        torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler.mark("start")
    t0.record(stream)
    steps(K)
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

    # --- distribution: 64 windows of one rotation each ---
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(N_WINDOWS + 1)]
    evs[0].record(stream)
    for w in range(N_WINDOWS):
        steps(n_sets)
        evs[w + 1].record(stream)
    torch.cuda.synchronize()
    win_us = [evs[w].elapsed_time(evs[w + 1]) * 1e3 / n_sets for w in range(N_WINDOWS)]

    # --- cold single calls: a 512 MiB scratch write before each, outside the window ---
    scratch = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    cold_us = []
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for i in range(N_COLD):
        scratch.fill_(i & 0xFF)
        c0.record(stream)
        sets[i % n_sets].call(handle, flags)
        c1.record(stream)
        torch.cuda.synchronize()
        cold_us.append(c0.elapsed_time(c1) * 1e3)
    del scratch

    # --- the same back-to-back steps without the early reads (decode only) ---
    plain_ms = None
    if kind != "prefill" and flags != 0:
        torch.cuda.synchronize()
        p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        p0.record(stream)
        steps(K, fl=0)
        p1.record(stream)
        torch.cuda.synchronize()
        plain_ms = max_over_ranks(p0.elapsed_time(p1), world, dev)

    # --- CUDA-graph replay: one graph holding one launch per set ---
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap):
        steps(n_sets, h=cap.cuda_stream)
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    reps = max(K // n_sets, 1)
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for _ in range(reps):
        graph.replay()
    g1.record(stream)
    torch.cuda.synchronize()
    graph_us = max_over_ranks(g0.elapsed_time(g1), world, dev) * 1e3 / (reps * n_sets)

    # --- end to end through the public API with host buffers ---
    # every step: one pinned host-to-device copy of the step's inputs, the
    # call, and a device-to-host read of its output.  Copies run on their own
    # streams.  Steps go in groups of G = n_sets / 2 (two groups' sets in
    # flight): a group's inputs travel while the previous group computes and
    # its outputs travel back while the next one computes.  The compute stream
    # waits on events only at group boundaries, so the calls of a group follow
    # one another directly on the stream and each may start while the one
    # before it drains; events keep each set's buffers free until the group
    # that last used them has finished with them.
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    rt = CudaRuntime()
    hs, hu, hd = handle, up.cuda_stream, down.cuda_stream
    G = max(n_sets // 2, 1)
    n_groups = n_sets // G                              # groups whose sets are in flight at once
    h2d_done = [rt.event() for _ in range(n_groups)]
    run_done = [rt.event() for _ in range(n_groups)]
    d2h_done = [rt.event() for _ in range(n_groups)]
    used = [False] * n_groups
    e2e_next = [0]                                      # the next step to issue

    def e2e_group(count):
        s0 = e2e_next[0]
        grp = (s0 // G) % n_groups                      # the slot whose sets this group uses
        ks = [(s0 + j) % n_sets for j in range(count)]
        if used[grp]:
            rt.wait(hu, run_done[grp])                  # the sets' inputs were consumed
        for k in ks:
            st = sets[k]
            rt.copy(st.packed.dev.data_ptr(), st.packed.host.data_ptr(), st.packed.total, rt.H2D, hu)
        rt.record(h2d_done[grp], hu)
        rt.wait(hs, h2d_done[grp])
        if used[grp]:
            rt.wait(hs, d2h_done[grp])                  # the sets' previous outputs were read back
        # the inputs were written by copies that the stream waited for, not
        # by the preceding kernel, so the early reads stay valid
        for k in ks:
            sets[k].call(hs, flags)
        rt.record(run_done[grp], hs)
        rt.wait(hd, run_done[grp])
        for k in ks:
            st = sets[k]
            rt.copy(st.host_out.data_ptr(), st.out.data_ptr(), st.out.numel() * st.out.element_size(), rt.D2H, hd)
        rt.record(d2h_done[grp], hd)
        used[grp] = True
        e2e_next[0] += count

    def e2e_run(steps_total):
        # groups start at multiples of G so that a group's sets are always the
        # same slot's; the first group may be shorter to get there
        done = 0
        while done < steps_total:
            s0 = e2e_next[0]
            count = min(G - s0 % G, steps_total - done)
            e2e_group(count)
            done += count

    def e2e_drain():
        for g in range(n_groups):
            if used[g]:
                rt.wait(hs, d2h_done[g])

    e2e_run(max(3, G))
    e2e_drain()
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    up.wait_event(e0)
    down.wait_event(e0)
    e2e_run(K)
    e2e_drain()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    h2d = sum(sets[s % n_sets].packed.total for s in range(K)) // K
    d2h = sum(sets[s % n_sets].out.numel() * 2 for s in range(K)) // K

    if rank != 0:
        return
    ms_per_step = elapsed_ms / K
    hbm_peak, tensor_peak, peak_kind = measured_peaks()
    bytes_per_step = bytes_k / K
    achieved = bytes_per_step / (ms_per_step * 1e-3) / 1e9
    cpu = cpu_baseline(name, case0)
    sd_name = synth.STATE_NAMES[case0.state_dtype]
    metric, unit = metric_unit(name)
    cpu["unit"] = unit
    line = {
        "metric": metric,
        "value": whole_job_value(updates_k / K, world, elapsed_ms, K),
        "unit": unit,
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "us_per_step": ms_per_step * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if (kind == "prefill" and args.prefill_form == "chunked") else "f32",
        "data": "synthetic",
        "config": {
            "workload": f"{name}: {WORKLOADS[name][0]}",
            "global_batch": case0.batch * world,
            "seq_len": draft_depth(name),
            "parallelism": f"independent batches, {world} GPU(s)",
            "state_dtype": sd_name,
            "flags": flags,
            "cache": f"inputs larger than L2: {n_sets} rotating input sets (token rows, index tables, disjoint "
                     f"state slots of a {num_slots}-slot pool); a step's bytes were last touched "
                     f">= {(n_sets - 1) * bytes_per_step / 1e6:.0f} MB of traffic earlier",
        },
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak,
                     "traffic": profiled_traffic(name) if (kind != "prefill" or args.prefill_form == "chunked")
                     else None,
                     "peak_kind": f"{peak_kind} HBM copy bandwidth",
                     "algorithmic_bytes_per_launch": bytes_per_step},
        "distribution": {
            "window_us": {"median": pct(win_us, 50), "p10": pct(win_us, 10), "p90": pct(win_us, 90),
                          "windows": N_WINDOWS, "steps_per_window": n_sets},
            "cold_call_us": {"median": pct(cold_us, 50), "p10": pct(cold_us, 10), "p90": pct(cold_us, 90),
                             "calls": N_COLD, "flush_bytes": FLUSH_BYTES},
        },
        "cpu_baseline": cpu,
        "e2e": {"value": whole_job_value(updates_k / K, world, e2e_ms, K), "unit": unit,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "graph_replay": {"value": updates_k / K * world / (graph_us * 1e-6), "unit": unit,
                         "us_per_step": graph_us},
        "gpu_launches": K,
        "clocks": clocks,
    }
    if plain_ms is not None:
        line["no_early_reads"] = {"us_per_step": plain_ms * 1e3 / K,
                                  "value": whole_job_value(updates_k / K, world, plain_ms, K)}
    if kind == "prefill":
        line["config"]["form"] = args.prefill_form
        if args.prefill_form == "chunked":
            tf = flops_k / K / (ms_per_step * 1e-3) / 1e12
            line["roofline_tensor"] = {"bound": "tensor", "achieved": tf, "peak": tensor_peak, "unit": "TFLOP/s",
                                       "frac": tf / tensor_peak, "peak_kind": f"{peak_kind} bf16 dense (burst)",
                                       "algorithmic_flops_per_launch": flops_k / K}
    elif kind == "decode":
        line["split"] = gdn.binding.chosen_split(sets[0].prepared.dims, case0.state_dtype)
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="bs32_t8_bf16")
    ap.add_argument("--split", type=lambda x: int(x, 0), default=0,
                    help="decode workloads: dims.split (0 = the library's choice; 1, 2, 4, 8, 0x102, 0x104, 0x201, 0x202)")
    ap.add_argument("--flags", type=lambda x: int(x, 0), default=GDN_PRE_INDEX | GDN_PRE_TOKENS | GDN_PRE_STATE,
                    help="decode and conv workloads: dims.flags (default 7 = GDN_PRE_INDEX | GDN_PRE_TOKENS | "
                         "GDN_PRE_STATE: the resident inputs and the rotating sets' disjoint state and conv slots are "
                         "not written by the preceding step)")
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
        run_gpu(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()

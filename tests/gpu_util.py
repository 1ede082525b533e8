"""GPU-side helpers for the parity tests: move a synthetic case to the device,
run the CUDA path through the C-ABI binding, run the oracle on the same
inputs, and compare."""
from __future__ import annotations

import numpy as np
import torch

import gated_deltanet_linear_sm_gb300 as gdn
from gated_deltanet_linear_sm_gb300 import synth
from oracle import oracle as orc
from tests.util import bf16_values, initial_pool, rel_l2, state_values

TORCH_STATE = {synth.F32: torch.float32, synth.BF16: torch.bfloat16, synth.F16: torch.float16}
OUT_SENTINEL = 0x7FBF          # a NaN bf16 pattern no kernel output can have


def t_bf16(bits, device):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def t_state(bits, state_dtype, device):
    arr = np.ascontiguousarray(bits)
    if state_dtype == synth.F32:
        return torch.from_numpy(arr).to(device)
    return torch.from_numpy(arr.view(np.int16)).to(device).view(TORCH_STATE[state_dtype])


def to_host_bits(t):
    if t.dtype == torch.float32:
        return t.cpu().numpy()
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def device_tensors(case, device):
    d = dict(
        q=t_bf16(case.q, device), k=t_bf16(case.k, device), v=t_bf16(case.v, device),
        a=t_bf16(case.a, device), b=t_bf16(case.b, device),
        z=t_bf16(case.z, device) if case.z is not None else None,
        A_log=torch.from_numpy(case.A_log).to(device),
        dt_bias=t_bf16(case.dt_bias, device),
        norm_w=t_bf16(case.norm_w, device) if case.norm_w is not None else None,
        state_indices=torch.from_numpy(case.state_indices).to(device),
        num_accepted=torch.from_numpy(case.num_accepted).to(device),
        cu_seqlens=torch.from_numpy(case.cu_seqlens).to(device),
        spec_token_indx=(torch.from_numpy(case.spec_token_indx).to(device)
                         if case.spec_token_indx is not None else None),
    )
    return d


def make_pool(case, device, seed=1234, slots=None):
    """Device pool: background slots hold random values from torch's device
    RNG (nobody compares them with the oracle; they only have to stay
    bit-identical), and ``slots`` (default: every slot the step touches) hold
    the generator's values."""
    shape = (case.num_slots, case.H_v, case.K, case.V)
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    pool = torch.randn(shape, generator=g, device=device, dtype=TORCH_STATE[case.state_dtype])
    touched = case.touched_slots() if slots is None else np.asarray(slots, dtype=np.int64)
    for start in range(0, len(touched), 256):
        chunk = touched[start:start + 256]
        vals = t_state(case.slot_values(chunk), case.state_dtype, device)
        pool[torch.from_numpy(chunk).to(device)] = vals
    return pool


def run_gpu(case, device, pool=None, *, split=0, flags=0, out=None, status=True, tensors=None, stream=None):
    """Run the CUDA path; returns (out, pool, status_word)."""
    t = tensors if tensors is not None else device_tensors(case, device)
    if pool is None:
        pool = make_pool(case, device)
    if out is None:
        out = torch.full((case.num_tokens, case.H_v, case.V), OUT_SENTINEL, dtype=torch.int16,
                         device=device).view(torch.bfloat16)
    st = torch.zeros(1, dtype=torch.int32, device=device) if status else None
    gdn.gdn_spec_decode(t["q"], t["k"], t["v"], t["a"], t["b"], t["z"], t["A_log"], t["dt_bias"],
                        t["norm_w"], pool, t["state_indices"], t["num_accepted"], t["cu_seqlens"], out,
                        spec_token_indx=t["spec_token_indx"], scale=case.scale, eps=case.eps,
                        max_T=case.max_T, split=split, flags=flags, status=st, stream=stream)
    return out, pool, st


def written_slots(case):
    ql = case.q_lens()
    rs = case.read_slots()
    s = set()
    for i in range(case.batch):
        if ql[i] <= 0 or rs[i] < 0 or rs[i] >= case.num_slots:
            continue
        for t in range(int(ql[i])):
            w = int(case.state_indices[i, t])
            if 0 <= w < case.num_slots:
                s.add(w)
    return np.array(sorted(s), dtype=np.int64)


def active_rows(case):
    ql = case.q_lens()
    rs = case.read_slots()
    rows = case.token_rows()
    out = []
    for i in range(case.batch):
        if ql[i] > 0 and 0 <= rs[i] < case.num_slots:
            out.extend(rows[case.cu_seqlens[i]:case.cu_seqlens[i + 1]].tolist())
    return np.array(sorted(out), dtype=np.int64)


def oracle_on(case, seqs=None, threads=None):
    """Oracle results for the whole case (compact pool) or for a subset of its
    sequences.  Returns (result dict, slot_map, rows, sub_case)."""
    import os
    if seqs is None:
        seqs = range(case.batch)
    sub, slot_map, rows = synth.subset(case, list(seqs))
    pool = initial_pool(sub, slot_map)
    res = orc.run_case(sub, pool, num_threads=threads or os.cpu_count() or 1)
    res["pool"] = pool
    return res, slot_map, rows, sub


def compare(case, out, pool, seqs=None, *, out_tol=5e-4, f32_state_tol=5e-4, narrow_tol=3e-2):
    """Compare the CUDA results with the oracle on the given sequences.
    Returns a dict of metrics; raises AssertionError on a tolerance miss."""
    res, slot_map, rows, sub = oracle_on(case, seqs)
    # outputs at the active rows of the selected sequences
    act = active_rows(sub)                        # sub-case row numbers
    metrics = {}
    if len(act):
        gpu_bits = out.view(torch.int16)[torch.from_numpy(rows[act]).to(out.device)].cpu().numpy().view(np.uint16)
        g = bf16_values(gpu_bits)
        want = bf16_values(res["out_bf16"][act])
        metrics["out_rel_l2"] = rel_l2(g, want)
        metrics["out_rel_l2_vs_f64"] = rel_l2(g, res["out_f64"][act])
        metrics["out_bits_equal"] = float(np.mean(gpu_bits == res["out_bf16"][act]))
        assert np.isfinite(g).all(), "non-finite output"
        assert metrics["out_rel_l2"] <= out_tol, metrics
    # written slots of the selected sequences
    wsub = written_slots(sub)
    if len(wsub):
        orig = slot_map[wsub]
        gpu = state_values(to_host_bits(pool[torch.from_numpy(orig).to(pool.device)]), case.state_dtype)
        want = state_values(res["pool"][wsub], case.state_dtype)
        metrics["state_rel_l2"] = rel_l2(gpu, want)
        metrics["state_max_abs"] = float(np.max(np.abs(gpu - want)))
        if case.state_dtype == synth.F32:
            assert metrics["state_rel_l2"] <= f32_state_tol, metrics
        else:
            bad = np.abs(gpu - want) > narrow_tol + narrow_tol * np.abs(want)
            metrics["state_bits_equal"] = float(np.mean(gpu == want))
            assert not bad.any(), (metrics, int(bad.sum()))
    return metrics

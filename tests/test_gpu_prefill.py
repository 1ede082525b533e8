"""Parity of the two prefill entry points (gdn_prefill, the per-token
recurrence, and gdn_prefill_chunked, the tensor-core chunked form; both
through the C-ABI) with the oracle's prefill routine: the same per-token step
over whole prompts, the state carried from a slot (or the zero state) and
stored once at the end (PR #52191 report, implementation steps 3-4).

Tolerances.  Both paths are held to the decode step's bounds (PR #51674
report, step 5: output rel L2 < 5e-4; FP32 state the same; narrow states
atol = rtol = 3e-2).  The recurrent path computes in FP32 like the decode
step.  The chunked path runs its products on the tensor cores at FP32
accuracy (PR #52191 report, step 4: the chunk products on FP32 buffers):
every operand is carried as a bf16 hi part and a bf16 lo part, so each
product is formed to about 2^-17 relative before FP32 accumulation.
"""
from __future__ import annotations

import dataclasses
import os

import numpy as np
import pytest
import torch

import gated_deltanet_linear_sm_gb300 as gdn
from gated_deltanet_linear_sm_gb300 import synth
from oracle import oracle as orc
from tests.gpu_util import OUT_SENTINEL, device_tensors, make_pool, to_host_bits
from tests.util import bf16_bits, bf16_values, rel_l2, state_values

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
THREADS = os.cpu_count() or 1

# entry point -> rel L2 bound for outputs and FP32 states
ENTRIES = {"recurrent": (gdn.gdn_prefill, 5e-4), "chunked": (gdn.gdn_prefill_chunked, 5e-4)}
ERRORS = []         # (test, entry, out rel L2, FP32-state rel L2), printed at the end of the module
WEAK_DECAY = (1e-3, 5e-2)


def _case(lens, sd, H_k=2, H_v=16, seed=50, gated=True, A_log_range=(1.0, 16.0)):
    return synth.make_case(batch=len(lens), H_k=H_k, H_v=H_v, T=max(lens), state_dtype=sd,
                           num_slots=max(4 * len(lens) + 8, 32), spec_stride=1, q_lens=list(lens),
                           acc=[1] * len(lens), gated=gated, A_log_range=A_log_range, seed=seed)


def _slots(case, seed, zero_every=3, skip_every=4, in_place=False):
    rng = np.random.default_rng(seed)
    perm = rng.permutation(case.num_slots).astype(np.int32)
    B = case.batch
    reads = perm[:B].copy()
    writes = reads.copy() if in_place else perm[B:2 * B].copy()
    if not in_place:
        reads[::zero_every] = -1          # zero initial state
        writes[1::skip_every] = -1        # no final write
    return reads, writes


def _run(entry, case, reads, writes):
    fn = ENTRIES[entry][0]
    pool_slots = sorted({int(s) for s in np.concatenate([reads, writes]) if s >= 0})
    pool = make_pool(case, DEV, slots=pool_slots)
    host = to_host_bits(pool)
    t = device_tensors(case, DEV)
    out = torch.full((case.num_tokens, case.H_v, case.V), OUT_SENTINEL, dtype=torch.int16,
                     device=DEV).view(torch.bfloat16)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    fn(t["q"], t["k"], t["v"], t["a"], t["b"], t["z"], t["A_log"], t["dt_bias"], t["norm_w"],
       pool, torch.from_numpy(reads).to(DEV), torch.from_numpy(writes).to(DEV), t["cu_seqlens"],
       out, scale=case.scale, eps=case.eps, status=st)
    torch.cuda.synchronize()
    ref = orc.prefill(q=case.q, k=case.k, v=case.v, a=case.a, b=case.b, z=case.z, A_log=case.A_log,
                      dt_bias=case.dt_bias, norm_w=case.norm_w, pool=host, state_dtype=case.state_dtype,
                      cu_seqlens=case.cu_seqlens, read_slots=reads, write_slots=writes, scale=case.scale,
                      eps=case.eps, num_threads=THREADS)
    return out, pool, st, ref, host


def _check(entry, case, out, pool, st, ref, host, writes):
    tol = ENTRIES[entry][1]
    assert int(st.item()) == 0
    g = bf16_values(out.view(torch.int16).cpu().numpy().view(np.uint16))
    w = bf16_values(ref["out_bf16"])
    assert np.all(np.isfinite(g))
    err_out = rel_l2(g, w)
    err_state = None
    if case.state_dtype == synth.F32:
        wr0 = [int(s) for s in writes if s >= 0]
        err_state = rel_l2(state_values(to_host_bits(pool), case.state_dtype)[wr0], state_values(host, case.state_dtype)[wr0])
    ERRORS.append((os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0], entry, err_out, err_state))
    assert err_out < tol, err_out
    gp = state_values(to_host_bits(pool), case.state_dtype)
    wp = state_values(host, case.state_dtype)
    wr = [int(s) for s in writes if s >= 0]
    others = np.setdiff1d(np.arange(case.num_slots), wr)
    # slots nobody writes stay bit-identical
    assert np.array_equal(to_host_bits(pool)[others], host[others])
    if case.state_dtype == synth.F32:
        err_state = rel_l2(gp[wr], wp[wr])
        assert err_state < tol, err_state
    else:
        assert np.all(np.abs(gp[wr] - wp[wr]) <= 3e-2 + 3e-2 * np.abs(wp[wr]))


@pytest.mark.parametrize("sd", [synth.F32, synth.BF16, synth.F16])
@pytest.mark.parametrize("entry", list(ENTRIES))
def test_ragged_prompts(entry, sd):
    """Prompt lengths across the 8-token rounds and the 64-token chunks (1, 7,
    9, 63, 64, 65, 130, 200), zero and slot initial states, some final writes
    skipped."""
    case = _case([1, 7, 9, 63, 64, 65, 130, 200], sd)
    reads, writes = _slots(case, 1)
    _check(entry, case, *_run(entry, case, reads, writes), writes)


@pytest.mark.parametrize("sd", [synth.F32, synth.BF16, synth.F16])
@pytest.mark.parametrize("entry", list(ENTRIES))
def test_ragged_prompts_few_units(entry, sd):
    """The same prompt lengths over 64 (sequence, v-head) units, fewer than
    half the SMs: the chunked form splits each unit's value columns over a
    2-CTA cluster (the test above, with 128 units, runs one CTA per unit)."""
    case = _case([1, 7, 9, 63, 64, 65, 130, 200], sd, H_k=1, H_v=8, seed=62)
    reads, writes = _slots(case, 9)
    _check(entry, case, *_run(entry, case, reads, writes), writes)


@pytest.mark.parametrize("H_k,ratio,lens", [
    (3, 1, [37, 70, 5]),                                          # 9 units: 2-CTA clusters
    (3, 4, [37, 70, 5]),                                          # 36 units
    (4, 2, [37, 70, 5, 64, 1, 100, 9, 20, 33, 65, 2, 128]),      # 96 units: one CTA per unit
], ids=["ratio1", "ratio4", "ratio2-96-units"])
@pytest.mark.parametrize("entry", list(ENTRIES))
def test_head_ratios(entry, H_k, ratio, lens):
    """v-heads per key head other than 8 (H_v = ratio H_k, v-head h reads key
    head h / ratio), FP32 state, in both launch forms of the chunked entry."""
    case = _case(lens, synth.F32, H_k=H_k, H_v=H_k * ratio, seed=63 + ratio)
    reads, writes = _slots(case, 10 + ratio)
    _check(entry, case, *_run(entry, case, reads, writes), writes)


@pytest.mark.parametrize("sd", [synth.F32, synth.BF16])
@pytest.mark.parametrize("entry", list(ENTRIES))
def test_long_prompts_weak_decay(entry, sd):
    """Decays close to 1 keep the state alive across many chunks, so every
    chunk-to-chunk carry shows in the outputs and the final state."""
    case = _case([1024, 333], sd, H_k=1, H_v=8, seed=56, A_log_range=WEAK_DECAY)
    reads, writes = _slots(case, 4, zero_every=2, skip_every=5)
    _check(entry, case, *_run(entry, case, reads, writes), writes)


@pytest.mark.parametrize("entry", list(ENTRIES))
def test_in_place_update(entry):
    case = _case([5, 33, 70], synth.BF16, seed=51)
    reads, writes = _slots(case, 2, in_place=True)
    _check(entry, case, *_run(entry, case, reads, writes), writes)


@pytest.mark.parametrize("entry", list(ENTRIES))
def test_ungated_raw_output(entry):
    case = _case([10, 90], synth.F32, H_k=1, H_v=8, seed=52, gated=False, A_log_range=WEAK_DECAY)
    reads, writes = _slots(case, 3)
    _check(entry, case, *_run(entry, case, reads, writes), writes)


@pytest.mark.parametrize("entry", list(ENTRIES))
def test_extreme_decay_stays_finite(entry):
    """g of several hundred per token: e^G underflows to zero inside a chunk,
    and every factor the chunked form uses is e^(non-positive)."""
    case = _case([3, 100], synth.F32, H_k=1, H_v=8, seed=57, A_log_range=(200.0, 400.0))
    reads, writes = _slots(case, 5, zero_every=7)
    _check(entry, case, *_run(entry, case, reads, writes), writes)


@pytest.mark.parametrize("entry", list(ENTRIES))
def test_prefill_then_speculative_step(entry):
    """The state a prefill stores is where the next speculative step rewinds
    to: prefill, then a decode step reading the prefill's slots, against the
    oracle doing the same two calls."""
    pre = _case([30, 11, 70], synth.F32, H_k=1, H_v=8, seed=53)
    reads = np.array([-1, -1, -1], np.int32)
    writes = np.array([2, 5, 9], np.int32)
    out1, pool, st, ref1, host = _run(entry, pre, reads, writes)
    _check(entry, pre, out1, pool, st, ref1, host, writes)
    dec = synth.make_case(batch=3, H_k=1, H_v=8, T=3, state_dtype=synth.F32, num_slots=pre.num_slots,
                          acc=[1, 1, 1], seed=54)
    dec.state_indices = np.array([[2, 20, 21], [5, 22, 23], [9, 24, 25]], np.int32)
    t = device_tensors(dec, DEV)
    out2 = torch.zeros(dec.num_tokens, dec.H_v, dec.V, dtype=torch.bfloat16, device=DEV)
    gdn.gdn_spec_decode(t["q"], t["k"], t["v"], t["a"], t["b"], t["z"], t["A_log"], t["dt_bias"], t["norm_w"],
                        pool, t["state_indices"], t["num_accepted"], t["cu_seqlens"], out2, max_T=3)
    torch.cuda.synchronize()
    ref2 = orc.run_case(dec, host)
    tol = ENTRIES[entry][1]
    g = bf16_values(out2.view(torch.int16).cpu().numpy().view(np.uint16))
    assert rel_l2(g, bf16_values(ref2["out_bf16"])) < tol
    w = dec.state_indices[:, :].ravel()
    assert rel_l2(pool[torch.from_numpy(w.astype(np.int64)).to(DEV)].cpu().numpy(), host[w]) < tol


@pytest.mark.parametrize("entry", list(ENTRIES))
def test_bad_slot_is_flagged_and_skipped(entry):
    fn = ENTRIES[entry][0]
    case = _case([6, 6, 6], synth.F32, H_k=1, H_v=8, seed=55)
    reads = np.array([1, case.num_slots + 3, 4], np.int32)
    writes = np.array([7, 8, 9], np.int32)
    pool = make_pool(case, DEV, slots=[1, 4])
    before = pool.clone()
    t = device_tensors(case, DEV)
    out = torch.zeros(case.num_tokens, case.H_v, case.V, dtype=torch.bfloat16, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    fn(t["q"], t["k"], t["v"], t["a"], t["b"], t["z"], t["A_log"], t["dt_bias"], t["norm_w"],
       pool, torch.from_numpy(reads).to(DEV), torch.from_numpy(writes).to(DEV), t["cu_seqlens"],
       out, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & gdn.binding.GDN_FLAG_SLOT_RANGE
    assert torch.equal(pool[8].view(torch.int32), before[8].view(torch.int32))
    assert not torch.equal(pool[7].view(torch.int32), before[7].view(torch.int32))


@pytest.mark.parametrize("entry", list(ENTRIES))
def test_empty_prompts_touch_nothing(entry):
    """Zero-length prompts between real ones: no output rows of theirs exist,
    their write slots stay as they were."""
    fn = ENTRIES[entry][0]
    case = _case([0, 20, 0, 5], synth.F32, H_k=1, H_v=8, seed=58)
    reads = np.array([1, 2, 3, 4], np.int32)
    writes = np.array([10, 11, 12, 13], np.int32)
    out, pool, st, ref, host = _run(entry, case, reads, writes)
    assert np.array_equal(to_host_bits(pool)[[10, 12]], host[[10, 12]])
    _check(entry, case, out, pool, st, ref, host, np.array([-1, 11, -1, 13], np.int32))


@pytest.mark.parametrize("bs,L", [(4, 1024), (32, 256)])
@pytest.mark.parametrize("entry", list(ENTRIES))
def test_benchmark_workloads_full_size(entry, bs, L):
    """The benchmark's prefill workloads at full size (H_k = 2, H_v = 16, bf16
    state, every prompt L tokens), started from slots and stored to other
    slots, every sequence compared."""
    case = synth.make_case(batch=bs, H_k=2, H_v=16, T=L, state_dtype=synth.BF16, num_slots=max(4 * bs, 64),
                           spec_stride=1, q_lens=[L] * bs, acc=[1] * bs, seed=59 + bs)
    reads, writes = _slots(case, 6, zero_every=10 ** 6, skip_every=10 ** 6)
    _check(entry, case, *_run(entry, case, reads, writes), writes)


@pytest.mark.parametrize("entry", list(ENTRIES))
def test_input_extremes(entry):
    """a + dt_bias above the softplus threshold (heads 0-3), beta saturated at 1
    and ~0 on alternate tokens, gates z at +-30, and rows whose q or k is zero
    (the L2-norm epsilon alone), across a chunk boundary."""
    case = _case([70, 5], synth.F32, H_k=1, H_v=8, seed=60)
    a, b, z = bf16_values(case.a), bf16_values(case.b), bf16_values(case.z)
    q, k = bf16_values(case.q), bf16_values(case.k)
    a[:, 0:4] = 30.0
    b[0::2, 4:8] = 40.0
    b[1::2, 4:8] = -40.0
    z[:, :, :64] = 30.0
    z[:, :, 64:] = -30.0
    q[3] = 0.0
    k[10] = 0.0
    k[64] = 0.0
    ext = dataclasses.replace(case, a=bf16_bits(a), b=bf16_bits(b), z=bf16_bits(z), q=bf16_bits(q), k=bf16_bits(k))
    reads, writes = _slots(ext, 7, zero_every=10 ** 6, skip_every=10 ** 6)
    _check(entry, ext, *_run(entry, ext, reads, writes), writes)


@pytest.mark.parametrize("lens", [[200, 65, 1], [200, 65, 1] * 30], ids=["2-cta-units", "1-cta-units"])
def test_chunked_runs_are_bit_identical(lens):
    """Two calls on the same inputs give the same out and pool bits (no
    atomics or order-dependent reductions in either launch form)."""
    case = _case(lens, synth.BF16, H_k=1, H_v=8, seed=70)
    reads, writes = _slots(case, 12, zero_every=10 ** 6, skip_every=10 ** 6)
    pool0 = make_pool(case, DEV, slots=sorted(s for s in set(reads.tolist()) | set(writes.tolist()) if s >= 0))
    t = device_tensors(case, DEV)
    res = []
    for _ in range(2):
        pool = pool0.clone()
        out = torch.zeros(case.num_tokens, case.H_v, case.V, dtype=torch.bfloat16, device=DEV)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        gdn.gdn_prefill_chunked(t["q"], t["k"], t["v"], t["a"], t["b"], t["z"], t["A_log"], t["dt_bias"],
                                t["norm_w"], pool, torch.from_numpy(reads).to(DEV), torch.from_numpy(writes).to(DEV),
                                t["cu_seqlens"], out, scale=case.scale, eps=case.eps, status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        res.append((out.view(torch.int16).clone(), pool.view(torch.int16).clone()))
    assert torch.equal(res[0][0], res[1][0]) and torch.equal(res[0][1], res[1][1])


@pytest.mark.parametrize("lens", [[200, 65, 1], [200, 65, 1] * 30], ids=["2-cta-units", "1-cta-units"])
def test_chunked_in_a_cuda_graph(lens):
    """The chunked prefill captured in a CUDA graph on a side stream (the
    2-CTA cluster launch included) and replayed gives the bits of a direct
    call."""
    case = _case(lens, synth.F32, H_k=1, H_v=8, seed=71)
    reads, writes = _slots(case, 13, zero_every=10 ** 6, skip_every=10 ** 6)
    pool0 = make_pool(case, DEV, slots=sorted(s for s in set(reads.tolist()) | set(writes.tolist()) if s >= 0))
    t = device_tensors(case, DEV)
    r_dev, w_dev = torch.from_numpy(reads).to(DEV), torch.from_numpy(writes).to(DEV)

    def call(pool, out, stream=None):
        gdn.gdn_prefill_chunked(t["q"], t["k"], t["v"], t["a"], t["b"], t["z"], t["A_log"], t["dt_bias"],
                                t["norm_w"], pool, r_dev, w_dev, t["cu_seqlens"], out, scale=case.scale,
                                eps=case.eps, stream=stream)

    direct_pool = pool0.clone()
    direct_out = torch.zeros(case.num_tokens, case.H_v, case.V, dtype=torch.bfloat16, device=DEV)
    call(direct_pool, direct_out)
    torch.cuda.synchronize()
    graph_pool = pool0.clone()
    graph_out = torch.zeros_like(direct_out)
    side = torch.cuda.Stream(DEV)
    side.wait_stream(torch.cuda.current_stream(DEV))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        call(graph_pool, graph_out, stream=side.cuda_stream)
    graph_pool.copy_(pool0)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(graph_out.view(torch.int16), direct_out.view(torch.int16))
    assert torch.equal(graph_pool.view(torch.int32), direct_pool.view(torch.int32))


@pytest.mark.parametrize("lens", [[100, 30], [100, 30] * 5], ids=["2-cta-units", "1-cta-units"])
def test_wait_timeout_is_flagged_and_the_next_launch_is_clean(lens):
    """A wait bound of one poll runs out on the first tensor-core wait: the
    call sets GDN_FLAG_TIMEOUT (and not GDN_FLAG_DRAIN: the products in flight
    finish under the default bound before tensor memory is released); with
    the default bound restored, the next launch matches the oracle.  16 units
    run as 2-CTA clusters (which go on to the last chunk), 80 units as one
    CTA each (which stop at once)."""
    case = _case(lens, synth.F32, H_k=1, H_v=8, seed=61)
    reads, writes = _slots(case, 8, zero_every=10 ** 6, skip_every=10 ** 6)
    pool = make_pool(case, DEV, slots=sorted(s for s in set(reads.tolist()) | set(writes.tolist()) if s >= 0))
    t = device_tensors(case, DEV)
    out = torch.zeros(case.num_tokens, case.H_v, case.V, dtype=torch.bfloat16, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    args = (t["q"], t["k"], t["v"], t["a"], t["b"], t["z"], t["A_log"], t["dt_bias"], t["norm_w"], pool.clone(),
            torch.from_numpy(reads).to(DEV), torch.from_numpy(writes).to(DEV), t["cu_seqlens"], out)
    gdn.binding.set_wait_limit(1)
    try:
        gdn.gdn_prefill_chunked(*args, status=st)
        torch.cuda.synchronize()
    finally:
        gdn.binding.set_wait_limit(0)
    flags = int(st.item())
    assert flags & gdn.binding.GDN_FLAG_TIMEOUT and not flags & gdn.binding.GDN_FLAG_DRAIN, flags
    _check("chunked", case, *_run("chunked", case, reads, writes), writes)


def test_zz_report_errors():
    """Prints the measured errors of every comparison above (run with -s)."""
    for name, entry, e_out, e_state in ERRORS:
        print(f"{entry:10s} out {e_out:.3e} state {e_state if e_state is None else f'{e_state:.3e}'}  {name}")

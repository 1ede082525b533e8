"""Parity of the CUDA path (through the C-ABI) with the FP64 oracle.

Tolerances (PR #51674 report, implementation step 5): outputs within relative
L2 5e-4 of the oracle's bf16-rounded output; fp32 state within relative L2
5e-4; bf16 / fp16 state within atol = rtol = 3e-2.  Which slots are written
and which bytes stay untouched is compared bit for bit.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

from gated_deltanet_linear_sm_gb300 import synth
from tests.gpu_util import (OUT_SENTINEL, active_rows, compare, device_tensors, make_pool, run_gpu,
                            to_host_bits, written_slots)
from tests.util import bf16_bits, bf16_values

pytestmark = pytest.mark.gpu

SPLITS = (1, 2, 4, 8, 0x102, 0x104, 0x201, 0x202)   # 0x100: GDN_SPLIT_NARROW (8 columns per warp); 0x200: GDN_SPLIT_HALFK


def _invariants(case, pool_before, pool_after, out):
    """Bit-exact slot routing: the changed slots are exactly the written ones
    (write-only slots were NaN-filled and must now be finite), and out rows
    outside the active spec rows keep the sentinel."""
    dt = torch.int32 if pool_before.dtype == torch.float32 else torch.int16
    changed = (pool_before.view(dt) != pool_after.view(dt)).flatten(1).any(1).cpu().numpy()
    w = written_slots(case)
    mask = np.zeros(case.num_slots, bool)
    mask[w] = True
    assert not (changed & ~mask).any(), "a slot outside the written set changed"
    assert torch.isfinite(pool_after[torch.from_numpy(w).to(pool_after.device)].float()).all()
    act = active_rows(case)
    rows = np.ones(case.num_tokens, bool)
    rows[act] = False
    untouched = out.view(torch.int16)[torch.from_numpy(np.nonzero(rows)[0]).to(out.device)]
    assert bool((untouched == OUT_SENTINEL).all()), "an out row outside the spec rows was written"


def _nan_write_only(case, pool):
    """Fill write-only slots with NaN so that a missed write is visible."""
    w = set(written_slots(case).tolist())
    r = set(int(s) for s in case.read_slots() if s >= 0)
    only = sorted(w - r)
    if only:
        pool[torch.tensor(only, device=pool.device)] = float("nan")


def _full_check(case, device, split, seqs=None):
    slots = None
    if seqs is not None:
        _, slots, _ = synth.subset(case, list(seqs))
    pool = make_pool(case, device, slots=slots)
    _nan_write_only(case, pool)
    before = pool.clone()
    out, pool, st = run_gpu(case, device, pool, split=split)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    _invariants(case, before, pool, out)
    return compare(case, out, pool, seqs)


@pytest.mark.parametrize("split", SPLITS)
def test_tiny(cuda_device, split):
    m = _full_check(synth.tiny(0), cuda_device, split)
    assert m["out_rel_l2"] < 5e-4


@pytest.mark.parametrize("split", SPLITS)
def test_decode_batch_bs32_t4_bf16(cuda_device, split):
    _full_check(synth.decode_batch(0), cuda_device, split)


@pytest.mark.parametrize("bs", [4, 8, 16, 32, 64, 128])
@pytest.mark.parametrize("sd", [synth.F32, synth.BF16])
def test_sweep_t8(cuda_device, bs, sd):
    """Batch sweep at full size (>= 2 GiB pool), automatic split (the launch
    the benchmark times).  Up to BS=32 every sequence is compared; above, a
    sample of 16 sequences (sequences are independent)."""
    case = synth.sweep(bs, sd)
    seqs = None if bs <= 32 else np.random.default_rng(bs).choice(bs, 16, replace=False)
    _full_check(case, cuda_device, 0, seqs)


@pytest.mark.parametrize("split", SPLITS)
def test_mixed_batch_gather_f16(cuda_device, split):
    """48 spec sequences among 80 non-spec rows, gathered through
    spec_token_indx, 10% padded slots, fp16 state."""
    _full_check(synth.mixed(0), cuda_device, split)


def test_large_bs256_sampled(cuda_device):
    """BS=256, H_k=4, H_v=32, T=8, bf16, 8192-slot (8 GiB) pool; 24 sampled
    sequences compared with the oracle, invariants over the whole pool."""
    case = synth.large(0)
    seqs = np.random.default_rng(7).choice(case.batch, 24, replace=False)
    _full_check(case, cuda_device, 0, seqs)


@pytest.mark.parametrize("sd", [synth.F32, synth.BF16, synth.F16])
@pytest.mark.parametrize("split", SPLITS)
def test_ragged_lengths_and_padding(cuda_device, sd, split):
    """Ragged q_len in {0..T} (q_len = 0 skipped), acceptance in {0..T}, 15%
    padded slots (a padded read slot skips the sequence), several tiles."""
    case = synth.make_case(batch=40, H_k=2, H_v=16, T=8, state_dtype=sd, num_slots=512,
                           q_lens="ragged", pad_prob=0.15, seed=21)
    _full_check(case, cuda_device, split)


@pytest.mark.parametrize("sd", [synth.F32, synth.BF16, synth.F16])
def test_ragged_padding_pipelined_writes(cuda_device, sd):
    """At most one CTA per SM (8 sequences x 16 v-heads) the slot writes are
    pipelined (a token's state is written during the next token): ragged
    q_len in {0..8}, 30% padded slots (skipped writes, padded sequences)."""
    case = synth.make_case(batch=8, H_k=2, H_v=16, T=8, state_dtype=sd, num_slots=128,
                           q_lens="ragged", pad_prob=0.3, seed=34)
    _full_check(case, cuda_device, 1)


@pytest.mark.parametrize("sd", [synth.BF16, synth.F16, synth.F32])
def test_single_token_steps(cuda_device, sd):
    """max_T = 1 (ordinary decode as a one-token step), every state dtype: 30 %
    padded slots, 640 units (more than one round of CTAs)."""
    case = synth.make_case(batch=40, H_k=2, H_v=16, T=1, state_dtype=sd, num_slots=256, pad_prob=0.3, seed=35)
    assert case.max_T == 1
    _full_check(case, cuda_device, 0)


@pytest.mark.parametrize("sd", [synth.BF16, synth.F16])
def test_single_token_flags_change_no_bit(cuda_device, sd):
    """One-token steps with ragged q_len in {0, 1}: the early-read flags change
    no bit of out or of the pool."""
    case = synth.make_case(batch=16, H_k=2, H_v=16, T=1, state_dtype=sd, num_slots=128, q_lens="ragged",
                           pad_prob=0.1, seed=36)
    pool0 = make_pool(case, cuda_device)
    res = []
    for flags in (0, 1, 3, 5, 7):
        out, pool, st = run_gpu(case, cuda_device, pool0.clone(), split=0, flags=flags)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        res.append((out.view(torch.int16).clone(), pool.view(torch.int16).clone()))
    for r in res[1:]:
        assert torch.equal(r[0], res[0][0]) and torch.equal(r[1], res[0][1])


@pytest.mark.parametrize("split", SPLITS)
def test_ungated_raw_readout(cuda_device, split):
    """z = norm_w = NULL: out is the raw readout o, which the RMSNorm would
    otherwise hide (it is nearly scale invariant)."""
    case = synth.make_case(batch=12, H_k=1, H_v=8, T=5, state_dtype=synth.F32, num_slots=128,
                           gated=False, seed=22)
    _full_check(case, cuda_device, split)


@pytest.mark.parametrize("ratio", [1, 4, 8])
def test_head_ratios(cuda_device, ratio):
    """Non-interleaved GQA for H_v = ratio * H_k (8 is the tuned case; the map
    is general)."""
    case = synth.make_case(batch=6, H_k=2, H_v=2 * ratio, T=3, state_dtype=synth.BF16, num_slots=64, seed=23)
    _full_check(case, cuda_device, 0)


def test_max_T_and_stride_larger_than_T(cuda_device):
    """spec_stride 8 with q_len up to 8 and max_T = 8; acceptance = 8 reads the
    last column."""
    case = synth.make_case(batch=9, H_k=1, H_v=8, T=8, state_dtype=synth.F32, num_slots=128,
                           acc=[8, 0, 1, 7, 8, 3, 2, 5, 8], seed=24)
    _full_check(case, cuda_device, 0)
    case = synth.make_case(batch=9, H_k=1, H_v=8, T=3, spec_stride=8, state_dtype=synth.F32,
                           num_slots=128, acc=[1, 2, 3, 0, 8, 5, 1, 1, 2], seed=25)
    _full_check(case, cuda_device, 0)


def test_ordinary_decode_identity(cuda_device):
    """T = 1, num_accepted = 1: read and write state_indices[i, 0] in place;
    equals the oracle's ordinary (non-speculative) decode."""
    from oracle import oracle as orc
    from tests.util import bf16_values, initial_pool
    case = synth.make_case(batch=20, H_k=2, H_v=16, T=1, state_dtype=synth.BF16, num_slots=64,
                           acc=[1] * 20, seed=26)
    out, pool, _ = run_gpu(case, cuda_device)
    hp = initial_pool(case)
    ref = orc.decode_nonspec(q=case.q, k=case.k, v=case.v, a=case.a, b=case.b, z=case.z,
                             A_log=case.A_log, dt_bias=case.dt_bias, norm_w=case.norm_w, pool=hp,
                             state_dtype=case.state_dtype, slots=case.state_indices[:, 0].copy())
    g = bf16_values(out.view(torch.int16).cpu().numpy().view(np.uint16))
    w = bf16_values(ref["out_bf16"])
    assert np.linalg.norm(g - w) / np.linalg.norm(w) < 5e-4
    s = case.state_indices[:, 0]
    gs = bf16_values(to_host_bits(pool[torch.from_numpy(s.astype(np.int64)).to(cuda_device)]))
    ws = bf16_values(hp[s])
    assert np.all(np.abs(gs - ws) <= 3e-2 + 3e-2 * np.abs(ws))


@pytest.mark.parametrize("flags", [0, 1, 3])
def test_two_steps_chain(cuda_device, flags):
    """Step 2 reads the slots step 1 wrote: two GPU calls in a row equal two
    oracle calls in a row (also with the index tables and token rows read
    before the dependency wait: the state still waits for step 1)."""
    from oracle import oracle as orc
    from tests.util import bf16_values, initial_pool
    case1 = synth.make_case(batch=8, H_k=1, H_v=8, T=4, state_dtype=synth.F32, num_slots=96, seed=27)
    case2 = synth.make_case(batch=8, H_k=1, H_v=8, T=4, state_dtype=synth.F32, num_slots=96, seed=28)
    # step 2 rewinds into step 1's slots: its slot table reuses step 1's table
    # for the read position and fresh slots elsewhere
    rng = np.random.default_rng(3)
    free = np.setdiff1d(np.arange(96), case1.state_indices.ravel())
    idx2 = rng.choice(free, size=case2.state_indices.shape, replace=False).astype(np.int32)
    for i in range(8):
        j = max(int(case2.num_accepted[i]) - 1, 0)
        idx2[i, j] = case1.state_indices[i, int(rng.integers(0, 4))]
    case2.state_indices = idx2
    pool = make_pool(case1, cuda_device)
    hp = initial_pool(case1)
    t2 = device_tensors(case2, cuda_device)               # step 2's inputs resident before step 1 runs
    out1, pool, _ = run_gpu(case1, cuda_device, pool, flags=flags)
    r1 = orc.run_case(case1, hp)
    out2, pool, _ = run_gpu(case2, cuda_device, pool, flags=flags, tensors=t2)
    r2 = orc.run_case(case2, hp)
    torch.cuda.synchronize()
    for out, r in ((out1, r1), (out2, r2)):
        g = bf16_values(out.view(torch.int16).cpu().numpy().view(np.uint16))
        w = bf16_values(r["out_bf16"])
        assert np.linalg.norm(g - w) / np.linalg.norm(w) < 5e-4
    w2 = written_slots(case2)
    gs = pool[torch.from_numpy(w2).to(cuda_device)].cpu().numpy().astype(np.float64)
    ws = hp[w2].astype(np.float64)
    assert np.linalg.norm(gs - ws) / np.linalg.norm(ws) < 5e-4


def test_packed_mixed_qkv_strides(cuda_device):
    """q, k, v passed as views into one packed [N, 2 H_k K + H_v V] tensor,
    a and b as views into one [N, 2 H_v] tensor (row strides through the ABI)."""
    import gated_deltanet_linear_sm_gb300 as gdn
    from tests.gpu_util import device_tensors
    case = synth.make_case(batch=10, H_k=2, H_v=16, T=4, state_dtype=synth.BF16, num_slots=128, seed=29)
    t = device_tensors(case, cuda_device)
    N, Hk, Hv, K = case.num_tokens, case.H_k, case.H_v, case.K
    packed = torch.cat([t["q"].reshape(N, -1), t["k"].reshape(N, -1), t["v"].reshape(N, -1)], 1).contiguous()
    ab = torch.cat([t["a"], t["b"]], 1).contiguous()
    q = packed[:, :Hk * K].view(N, Hk, K)
    k = packed[:, Hk * K:2 * Hk * K].view(N, Hk, K)
    v = packed[:, 2 * Hk * K:].view(N, Hv, K)
    assert q.stride(0) == packed.shape[1]
    pool = make_pool(case, cuda_device)
    out = torch.zeros(N, Hv, K, dtype=torch.bfloat16, device=cuda_device)
    gdn.gdn_spec_decode(q, k, v, ab[:, :Hv], ab[:, Hv:], t["z"], t["A_log"], t["dt_bias"], t["norm_w"],
                        pool, t["state_indices"], t["num_accepted"], t["cu_seqlens"], out, max_T=4)
    compare(case, out, pool)


@pytest.mark.parametrize("flags", [0, 3, 7])
def test_graph_capture_replays(cuda_device, flags):
    """A call captured in a CUDA graph and replayed gives the same bits as an
    eager call on the same inputs (the launch needs no host sync)."""
    import gated_deltanet_linear_sm_gb300 as gdn
    from tests.gpu_util import device_tensors
    case = synth.decode_batch(0)
    t = device_tensors(case, cuda_device)
    pool0 = make_pool(case, cuda_device)
    outs = []
    for mode in ("eager", "graph"):
        pool = pool0.clone()
        out = torch.zeros(case.num_tokens, case.H_v, case.V, dtype=torch.bfloat16, device=cuda_device)
        call = gdn.prepare(t["q"], t["k"], t["v"], t["a"], t["b"], t["z"], t["A_log"], t["dt_bias"],
                           t["norm_w"], pool, t["state_indices"], t["num_accepted"], t["cu_seqlens"], out,
                           flags=flags)
        if mode == "eager":
            call()
        else:
            s = torch.cuda.Stream(cuda_device)
            s.wait_stream(torch.cuda.current_stream(cuda_device))
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                call()
            g.replay()
        torch.cuda.synchronize()
        outs.append((out.clone(), pool.clone()))
    assert torch.equal(outs[0][0].view(torch.int16), outs[1][0].view(torch.int16))
    assert torch.equal(outs[0][1].view(torch.int16), outs[1][1].view(torch.int16))


def test_deterministic(cuda_device):
    case = synth.sweep(16, synth.BF16, num_slots=1024)
    r = []
    for _ in range(2):
        out, pool, _ = run_gpu(case, cuda_device)
        torch.cuda.synchronize()
        r.append((out.view(torch.int16).clone(), pool.view(torch.int16).clone()))
    assert torch.equal(r[0][0], r[1][0]) and torch.equal(r[0][1], r[1][1])


@pytest.mark.parametrize("split", [0, 0x102, 0x202])
def test_gate_and_input_extremes(cuda_device, split):
    """Each input at the end of its range, against the oracle: a + dt_bias above
    the softplus threshold (heads 0-3), per-token decays that underflow to 0
    (heads 4-7) or stay within 1e-4 of 1 (heads 8-11), beta saturated at 1 and
    at ~0 (heads 12-15, alternate tokens), output gates z at +-30, a zero q and
    k row (the L2-norm epsilon alone) and a state pool of std 30."""
    case = synth.make_case(batch=6, H_k=2, H_v=16, T=8, state_dtype=synth.F32, num_slots=128, seed=29)
    a, b, z = bf16_values(case.a), bf16_values(case.b), bf16_values(case.z)
    q, k = bf16_values(case.q), bf16_values(case.k)
    A_log = case.A_log.copy()
    a[:, 0:4] = 30.0
    A_log[4:8] = np.log(400.0)
    A_log[8:12] = np.log(1e-4)
    b[0::2, 12:16] = 40.0
    b[1::2, 12:16] = -40.0
    z[:, 0:8, :64] = 30.0
    z[:, 8:16, 64:] = -30.0
    q[0, 0] = 0.0
    k[0, 0] = 0.0
    ext = dataclasses.replace(case, a=bf16_bits(a), b=bf16_bits(b), z=bf16_bits(z), q=bf16_bits(q),
                              k=bf16_bits(k), A_log=A_log.astype(np.float32), pool_std=30.0)
    m = _full_check(ext, cuda_device, split)
    assert m["out_rel_l2"] < 5e-4


@pytest.mark.parametrize("split", [1, 2, 0x102, 0x201, 0x202])
@pytest.mark.parametrize("sd", [synth.F32, synth.BF16])
def test_early_read_flags_change_no_bit(cuda_device, sd, split):
    """GDN_PRE_INDEX, with GDN_PRE_TOKENS and / or GDN_PRE_STATE, moves reads
    ahead of the dependency wait; the results (out and every pool byte) are
    bit-identical to flags = 0, on a ragged, padded batch."""
    import gated_deltanet_linear_sm_gb300 as gdn
    case = synth.make_case(batch=24, H_k=2, H_v=16, T=8, state_dtype=sd, num_slots=400, q_lens="ragged",
                           pad_prob=0.1, seed=31)
    pool0 = make_pool(case, cuda_device)
    res = []
    for flags in (0, 1, 3, 5, 7):
        out, pool, st = run_gpu(case, cuda_device, pool0.clone(), split=split, flags=flags)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        dt = torch.int32 if sd == synth.F32 else torch.int16
        res.append((out.view(torch.int16).clone(), pool.view(dt).clone()))
    for r in res[1:]:
        assert torch.equal(r[0], res[0][0]) and torch.equal(r[1], res[0][1])


def test_early_state_reads_between_independent_steps(cuda_device):
    """GDN_PRE_STATE across back-to-back steps whose slots are disjoint (the
    second step's rewound slots were not written by the first): both match
    the oracle, as with flags = 0."""
    from oracle import oracle as orc
    from tests.util import bf16_values, initial_pool
    case1 = synth.make_case(batch=8, H_k=1, H_v=8, T=4, state_dtype=synth.F32, num_slots=96, seed=32)
    case2 = synth.make_case(batch=8, H_k=1, H_v=8, T=4, state_dtype=synth.F32, num_slots=96, seed=33)
    free = np.setdiff1d(np.arange(96), case1.state_indices.ravel())
    case2.state_indices = np.random.default_rng(4).choice(free, size=case2.state_indices.shape,
                                                          replace=False).astype(np.int32)
    pool = make_pool(case1, cuda_device, slots=np.union1d(case1.touched_slots(), case2.touched_slots()))
    hp = initial_pool(case1)
    hp[case2.touched_slots()] = case1.slot_values(case2.touched_slots())     # make_pool fills them so
    t2 = device_tensors(case2, cuda_device)
    out1, pool, _ = run_gpu(case1, cuda_device, pool, flags=7)
    out2, pool, _ = run_gpu(case2, cuda_device, pool, flags=7, tensors=t2)
    torch.cuda.synchronize()
    r1 = orc.run_case(case1, hp)
    r2 = orc.run_case(case2, hp)
    for out, r in ((out1, r1), (out2, r2)):
        g = bf16_values(out.view(torch.int16).cpu().numpy().view(np.uint16))
        w = bf16_values(r["out_bf16"])
        assert np.linalg.norm(g - w) / np.linalg.norm(w) < 5e-4

"""Parity of the prefill entry point (gdn_prefill, through the C-ABI) with the
oracle's prefill routine: the same per-token step over whole prompts, the
state carried from a slot (or the zero state) and stored once at the end
(PR #52191 report, implementation steps 3-4)."""
from __future__ import annotations

import os

import numpy as np
import pytest
import torch

import gated_deltanet_linear_sm_gb300 as gdn
from gated_deltanet_linear_sm_gb300 import synth
from oracle import oracle as orc
from tests.gpu_util import OUT_SENTINEL, TORCH_STATE, device_tensors, make_pool, to_host_bits
from tests.util import bf16_values, rel_l2, state_values

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
THREADS = os.cpu_count() or 1


def _case(lens, sd, H_k=2, H_v=16, seed=50, gated=True):
    return synth.make_case(batch=len(lens), H_k=H_k, H_v=H_v, T=max(lens), state_dtype=sd,
                           num_slots=max(4 * len(lens) + 8, 32), spec_stride=1, q_lens=list(lens),
                           acc=[1] * len(lens), gated=gated, seed=seed)


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


def _run(case, reads, writes):
    pool_slots = sorted({int(s) for s in np.concatenate([reads, writes]) if s >= 0})
    pool = make_pool(case, DEV, slots=pool_slots)
    host = to_host_bits(pool)
    t = device_tensors(case, DEV)
    out = torch.full((case.num_tokens, case.H_v, case.V), OUT_SENTINEL, dtype=torch.int16,
                     device=DEV).view(torch.bfloat16)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    gdn.gdn_prefill(t["q"], t["k"], t["v"], t["a"], t["b"], t["z"], t["A_log"], t["dt_bias"], t["norm_w"],
                    pool, torch.from_numpy(reads).to(DEV), torch.from_numpy(writes).to(DEV), t["cu_seqlens"],
                    out, scale=case.scale, eps=case.eps, status=st)
    torch.cuda.synchronize()
    ref = orc.prefill(q=case.q, k=case.k, v=case.v, a=case.a, b=case.b, z=case.z, A_log=case.A_log,
                      dt_bias=case.dt_bias, norm_w=case.norm_w, pool=host, state_dtype=case.state_dtype,
                      cu_seqlens=case.cu_seqlens, read_slots=reads, write_slots=writes, scale=case.scale,
                      eps=case.eps, num_threads=THREADS)
    return out, pool, st, ref, host


def _check(case, out, pool, st, ref, host, writes):
    assert int(st.item()) == 0
    g = bf16_values(out.view(torch.int16).cpu().numpy().view(np.uint16))
    w = bf16_values(ref["out_bf16"])
    assert rel_l2(g, w) < 5e-4
    gp = state_values(to_host_bits(pool), case.state_dtype)
    wp = state_values(host, case.state_dtype)
    wr = [int(s) for s in writes if s >= 0]
    others = np.setdiff1d(np.arange(case.num_slots), wr)
    # slots nobody writes stay bit-identical
    assert np.array_equal(to_host_bits(pool)[others], host[others])
    if case.state_dtype == synth.F32:
        assert rel_l2(gp[wr], wp[wr]) < 5e-4
    else:
        assert np.all(np.abs(gp[wr] - wp[wr]) <= 3e-2 + 3e-2 * np.abs(wp[wr]))


@pytest.mark.parametrize("sd", [synth.F32, synth.BF16, synth.F16])
def test_ragged_prompts(sd):
    """Prompt lengths across the 8-token rounds (1, 7, 8, 9, 17, 64, 200),
    zero and slot initial states, some final writes skipped."""
    case = _case([1, 7, 8, 9, 17, 64, 200], sd)
    reads, writes = _slots(case, 1)
    _check(case, *_run(case, reads, writes), writes)


def test_in_place_update():
    case = _case([5, 33, 12], synth.BF16, seed=51)
    reads, writes = _slots(case, 2, in_place=True)
    _check(case, *_run(case, reads, writes), writes)


def test_ungated_raw_output():
    case = _case([10, 25], synth.F32, H_k=1, H_v=8, seed=52, gated=False)
    reads, writes = _slots(case, 3)
    _check(case, *_run(case, reads, writes), writes)


def test_prefill_then_speculative_step():
    """The state a prefill stores is where the next speculative step rewinds
    to: prefill, then a decode step reading the prefill's slots, against the
    oracle doing the same two calls."""
    pre = _case([30, 11, 4], synth.F32, H_k=1, H_v=8, seed=53)
    reads = np.array([-1, -1, -1], np.int32)
    writes = np.array([2, 5, 9], np.int32)
    out1, pool, st, ref1, host = _run(pre, reads, writes)
    _check(pre, out1, pool, st, ref1, host, writes)
    dec = synth.make_case(batch=3, H_k=1, H_v=8, T=3, state_dtype=synth.F32, num_slots=pre.num_slots,
                          acc=[1, 1, 1], seed=54)
    dec.state_indices = np.array([[2, 20, 21], [5, 22, 23], [9, 24, 25]], np.int32)
    t = device_tensors(dec, DEV)
    out2 = torch.zeros(dec.num_tokens, dec.H_v, dec.V, dtype=torch.bfloat16, device=DEV)
    gdn.gdn_spec_decode(t["q"], t["k"], t["v"], t["a"], t["b"], t["z"], t["A_log"], t["dt_bias"], t["norm_w"],
                        pool, t["state_indices"], t["num_accepted"], t["cu_seqlens"], out2, max_T=3)
    torch.cuda.synchronize()
    ref2 = orc.run_case(dec, host)
    g = bf16_values(out2.view(torch.int16).cpu().numpy().view(np.uint16))
    assert rel_l2(g, bf16_values(ref2["out_bf16"])) < 5e-4
    w = dec.state_indices[:, :].ravel()
    assert rel_l2(pool[torch.from_numpy(w.astype(np.int64)).to(DEV)].cpu().numpy(), host[w]) < 5e-4


def test_bad_slot_is_flagged_and_skipped():
    case = _case([6, 6, 6], synth.F32, H_k=1, H_v=8, seed=55)
    reads = np.array([1, case.num_slots + 3, 4], np.int32)
    writes = np.array([7, 8, 9], np.int32)
    pool = make_pool(case, DEV, slots=[1, 4])
    before = pool.clone()
    t = device_tensors(case, DEV)
    out = torch.zeros(case.num_tokens, case.H_v, case.V, dtype=torch.bfloat16, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    gdn.gdn_prefill(t["q"], t["k"], t["v"], t["a"], t["b"], t["z"], t["A_log"], t["dt_bias"], t["norm_w"],
                    pool, torch.from_numpy(reads).to(DEV), torch.from_numpy(writes).to(DEV), t["cu_seqlens"],
                    out, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & gdn.binding.GDN_FLAG_SLOT_RANGE
    assert torch.equal(pool[8].view(torch.int32), before[8].view(torch.int32))
    assert not torch.equal(pool[7].view(torch.int32), before[7].view(torch.int32))

"""Bad DEVICE data is skipped and reported through the status word, never
trapped (PR #46090 report, review highlights: spec_state_indices was left
unvalidated).  Every case below is one the kernel range-checks before any
access; the other sequences of the batch must still match the oracle."""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

import gated_deltanet_linear_sm_gb300 as gdn
from gated_deltanet_linear_sm_gb300 import synth
from tests.gpu_util import OUT_SENTINEL, compare, device_tensors, make_pool, run_gpu

pytestmark = pytest.mark.gpu

BAD = 3            # the corrupted sequence


def _base():
    return synth.make_case(batch=8, H_k=1, H_v=8, T=4, state_dtype=synth.F32, num_slots=64,
                           acc=[1, 2, 3, 4, 0, 1, 2, 3], seed=31)


def _rows_of(case, i):
    return case.token_rows()[case.cu_seqlens[i]:case.cu_seqlens[i + 1]]


def _run_and_check(case, gpu_case, flag, skipped_seq=True, expect=None, split=0, flags=0):
    """Run gpu_case (the corrupted one); compare every other sequence with the
    oracle on `expect` (default: case), check the flag and that the corrupted
    sequence left its slots and rows alone."""
    dev = torch.device("cuda", 0)
    pool = make_pool(case, dev)
    before = pool.clone()
    out, pool, st = run_gpu(gpu_case, dev, pool, split=split, flags=flags)
    torch.cuda.synchronize()
    assert int(st.item()) & flag, int(st.item())
    good = [i for i in range(case.batch) if not (skipped_seq and i == BAD)]
    compare(expect or case, out, pool, good)
    if skipped_seq:
        for s in case.state_indices[BAD]:
            if 0 <= s < case.num_slots:
                assert torch.equal(pool[int(s)].view(torch.int32), before[int(s)].view(torch.int32))
        rows = torch.from_numpy(_rows_of(case, BAD).astype(np.int64)).to(dev)
        assert bool((out.view(torch.int16)[rows] == OUT_SENTINEL).all())


@pytest.mark.parametrize("split", [1, 8, 0x102, 0x202])
def test_num_accepted_beyond_stride(split):
    case = _base()
    bad = dataclasses.replace(case, num_accepted=case.num_accepted.copy())
    bad.num_accepted[BAD] = case.spec_stride + 1
    _run_and_check(case, bad, gdn.binding.GDN_FLAG_ACCEPTED, split=split)


@pytest.mark.parametrize("flags", [1, 3])
def test_bad_data_with_early_reads(flags):
    """The exits taken on bad index data come before the dependency wait when
    the index tables are read early; each still waits before it reports."""
    case = _base()
    bad = dataclasses.replace(case, num_accepted=case.num_accepted.copy(), state_indices=case.state_indices.copy())
    bad.num_accepted[BAD] = case.spec_stride + 1
    _run_and_check(case, bad, gdn.binding.GDN_FLAG_ACCEPTED, flags=flags)
    bad = dataclasses.replace(case, state_indices=case.state_indices.copy())
    bad.state_indices[BAD, max(int(case.num_accepted[BAD]) - 1, 0)] = case.num_slots + 7
    _run_and_check(case, bad, gdn.binding.GDN_FLAG_SLOT_RANGE, flags=flags)


@pytest.mark.parametrize("split", [1, 8, 0x102, 0x202])
def test_read_slot_out_of_range(split):
    case = _base()
    bad = dataclasses.replace(case, state_indices=case.state_indices.copy())
    j = max(int(case.num_accepted[BAD]) - 1, 0)
    bad.state_indices[BAD, j] = case.num_slots + 5
    _run_and_check(case, bad, gdn.binding.GDN_FLAG_SLOT_RANGE, split=split)


def test_write_slot_out_of_range_skips_only_that_write():
    case = _base()
    j = max(int(case.num_accepted[BAD]) - 1, 0)
    t = (j + 1) % 4                                   # a write-only position
    bad = dataclasses.replace(case, state_indices=case.state_indices.copy())
    bad.state_indices[BAD, t] = case.num_slots + 1
    expect = dataclasses.replace(case, state_indices=case.state_indices.copy())
    expect.state_indices[BAD, t] = -1                 # the oracle: that write skipped
    _run_and_check(case, bad, gdn.binding.GDN_FLAG_SLOT_RANGE, skipped_seq=False, expect=expect)


def test_q_len_beyond_max_T():
    case = _base()
    lens = np.full(case.batch, 2)
    lens[BAD] = 4
    c2 = synth.make_case(batch=8, H_k=1, H_v=8, T=4, state_dtype=synth.F32, num_slots=64,
                         q_lens=lens, acc=[1, 2, 1, 4, 0, 1, 2, 1], seed=32)
    gpu_case = dataclasses.replace(c2, max_T=2)       # the host bound is wrong for sequence BAD
    _run_and_check(c2, gpu_case, gdn.binding.GDN_FLAG_QLEN)


@pytest.mark.parametrize("split", [1, 4, 0x104, 0x201])
def test_gathered_row_out_of_range(split):
    case = synth.make_case(batch=8, H_k=1, H_v=8, T=4, state_dtype=synth.F32, num_slots=64,
                           extra_rows=5, acc=[1, 2, 3, 4, 0, 1, 2, 3], seed=33)
    bad = dataclasses.replace(case, spec_token_indx=case.spec_token_indx.copy())
    bad.spec_token_indx[case.cu_seqlens[BAD] + 2] = case.num_tokens + 7
    _run_and_check(case, bad, gdn.binding.GDN_FLAG_TOKEN_ROW, split=split)


def test_cu_seqlens_beyond_total():
    """cu_seqlens[i+1] > cu_seqlens[batch] (non-monotone table): positions past
    the end of spec_token_indx are never read."""
    case = synth.make_case(batch=8, H_k=1, H_v=8, T=4, state_dtype=synth.F32, num_slots=64,
                           q_lens=[4, 4, 4, 4, 4, 4, 4, 0], extra_rows=3, seed=34)
    dev = torch.device("cuda", 0)
    t = device_tensors(case, dev)
    cu = case.cu_seqlens.copy()
    cu[-1] = cu[-3]                                   # total shrinks: sequence 6 now ends past it
    t["cu_seqlens"] = torch.from_numpy(cu).to(dev)
    pool = make_pool(case, dev)
    out, pool, st = run_gpu(case, dev, pool, tensors=t)
    torch.cuda.synchronize()
    assert int(st.item()) & gdn.binding.GDN_FLAG_TOKEN_ROW
    compare(case, out, pool, [0, 1, 2, 3, 4, 5])


def test_no_status_word_is_fine():
    case = _base()
    bad = dataclasses.replace(case, num_accepted=case.num_accepted.copy())
    bad.num_accepted[BAD] = 99
    dev = torch.device("cuda", 0)
    out, pool, st = run_gpu(bad, dev, make_pool(case, dev), status=False)
    torch.cuda.synchronize()
    assert st is None
    compare(case, out, pool, [i for i in range(case.batch) if i != BAD])


def test_bad_units_among_many():
    """1,024 units (64 sequences x 16 v-heads), more than the GPU holds at
    once, so the CTAs run in several waves.  Sequence BAD has a read slot out
    of range and sequence 40 a gathered row out of range: both are skipped
    and flagged, and every other unit, before and after them, still matches
    the oracle."""
    case = synth.make_case(batch=64, H_k=2, H_v=16, T=8, state_dtype=synth.BF16, num_slots=1100,
                           extra_rows=9, seed=35)
    bad = dataclasses.replace(case, state_indices=case.state_indices.copy(),
                              spec_token_indx=case.spec_token_indx.copy())
    j = max(int(case.num_accepted[BAD]) - 1, 0)
    bad.state_indices[BAD, j] = case.num_slots + 5
    bad.spec_token_indx[case.cu_seqlens[40] + 1] = case.num_tokens + 3
    dev = torch.device("cuda", 0)
    pool = make_pool(case, dev)
    before = pool.clone()
    out, pool, st = run_gpu(bad, dev, pool)
    torch.cuda.synchronize()
    flags = int(st.item())
    assert flags & gdn.binding.GDN_FLAG_SLOT_RANGE and flags & gdn.binding.GDN_FLAG_TOKEN_ROW, flags
    compare(case, out, pool, [i for i in range(case.batch) if i not in (BAD, 40)])
    for i in (BAD, 40):
        for s in case.state_indices[i]:
            if 0 <= s < case.num_slots:
                assert torch.equal(pool[int(s)].view(torch.int16), before[int(s)].view(torch.int16))
        rows = torch.from_numpy(_rows_of(case, i).astype(np.int64)).to(dev)
        assert bool((out.view(torch.int16)[rows] == OUT_SENTINEL).all())

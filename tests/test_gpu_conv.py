"""Parity of gdn_spec_decode_conv (the speculative step with the short causal
convolution and its rewind fused in front, through the C-ABI) with the
oracle's gdn_oracle_spec_decode_conv on the same seeded inputs.

Outputs and written state slots use the decode step's bounds (PR #51674
report, step 5: output rel L2 < 5e-4, FP32 state the same, narrow states
atol = rtol = 3e-2); the new conv slots hold copied input bits, so they must
match bit for bit, and every other conv slot must be untouched."""
from __future__ import annotations

import os

import numpy as np
import pytest
import torch

import gated_deltanet_linear_sm_gb300 as gdn
from gated_deltanet_linear_sm_gb300 import synth
from oracle import oracle as orc
from tests.gpu_util import OUT_SENTINEL, active_rows, make_pool, t_bf16, to_host_bits, written_slots
from tests.util import bf16_values, rel_l2, state_values

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
THREADS = os.cpu_count() or 1


def _case(batch=6, T=8, sd=synth.BF16, H_k=2, H_v=16, seed=70, q_lens="ragged", **kw):
    return synth.make_case(batch=batch, H_k=H_k, H_v=H_v, T=T, state_dtype=sd, num_slots=2 * batch * T + 8,
                           q_lens=q_lens, seed=seed, **kw)


class Step:
    """One call on the GPU and the same call on the oracle, from the same pools."""

    def __init__(self, case, ci, pool=None, conv_pool=None):
        self.case, self.ci = case, ci
        self.pool = make_pool(case, DEV) if pool is None else pool
        self.host = to_host_bits(self.pool)
        self.before = self.host.copy()
        self.conv = t_bf16(ci.pool, DEV) if conv_pool is None else conv_pool
        self.conv_host = self.conv.view(torch.int16).cpu().numpy().view(np.uint16).copy()
        self.conv_before = self.conv_host.copy()

    def run(self, conv_in=None, conv_out=None, flags=0):
        case, ci = self.case, self.ci
        conv_in = ci.conv_in if conv_in is None else conv_in
        conv_out = ci.conv_out if conv_out is None else conv_out
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
        self.out = torch.full((case.num_tokens, case.H_v, case.V), OUT_SENTINEL, dtype=torch.int16,
                              device=DEV).view(torch.bfloat16)
        self.status = torch.zeros(1, dtype=torch.int32, device=DEV)
        gdn.gdn_spec_decode_conv(
            t_bf16(ci.x, DEV), t_bf16(ci.weight, DEV), t_bf16(ci.bias, DEV) if ci.bias is not None else None,
            self.conv, t(conv_in), t(conv_out), t_bf16(case.a, DEV), t_bf16(case.b, DEV),
            t_bf16(case.z, DEV), t(case.A_log), t_bf16(case.dt_bias, DEV), t_bf16(case.norm_w, DEV), self.pool,
            t(case.state_indices), t(case.num_accepted), t(case.cu_seqlens), self.out, H_k=case.H_k,
            spec_token_indx=t(case.spec_token_indx) if case.spec_token_indx is not None else None,
            scale=case.scale, eps=case.eps, max_T=case.max_T, flags=flags, status=self.status)
        torch.cuda.synchronize()
        self.ref = orc.spec_decode_conv(
            x=ci.x, conv_weight=ci.weight, conv_bias=ci.bias, conv_pool=self.conv_host, conv_in=conv_in,
            conv_out=conv_out, H_k=case.H_k, K=case.K, a=case.a, b=case.b, z=case.z, A_log=case.A_log,
            dt_bias=case.dt_bias, norm_w=case.norm_w, pool=self.host, state_dtype=case.state_dtype,
            state_indices=case.state_indices, num_accepted=case.num_accepted, cu_seqlens=case.cu_seqlens,
            spec_token_indx=case.spec_token_indx, scale=case.scale, eps=case.eps, num_threads=THREADS)
        return self

    def check(self):
        case = self.case
        assert int(self.status.item()) == 0
        rows = active_rows(case)
        assert len(rows)
        g = bf16_values(self.out.view(torch.int16).cpu().numpy().view(np.uint16)[rows])
        assert np.isfinite(g).all()
        err = rel_l2(g, bf16_values(self.ref["out_bf16"][rows]))
        assert err < 5e-4, err
        ws = written_slots(case)
        gp = to_host_bits(self.pool)
        if len(ws):
            a = state_values(gp[ws], case.state_dtype)
            b = state_values(self.host[ws], case.state_dtype)
            if case.state_dtype == synth.F32:
                assert rel_l2(a, b) < 5e-4
            else:
                assert np.all(np.abs(a - b) <= 3e-2 + 3e-2 * np.abs(b))
        others = np.setdiff1d(np.arange(case.num_slots), ws)
        assert np.array_equal(gp[others], self.before[others])
        # conv slots: the new ones bit for bit, the rest untouched
        got = self.conv.view(torch.int16).cpu().numpy().view(np.uint16)
        assert np.array_equal(got, self.conv_host)
        return self


@pytest.mark.parametrize("width,bias", [(4, True), (4, False), (3, True), (2, True), (1, False)])
def test_widths_and_bias(width, bias):
    case = _case(seed=70 + width)
    ci = synth.conv_inputs(case, width=width, with_bias=bias, seed=width)
    Step(case, ci).run().check()


@pytest.mark.parametrize("sd", [synth.F32, synth.F16])
def test_state_dtypes(sd):
    case = _case(sd=sd, seed=80 + sd)
    Step(case, synth.conv_inputs(case, seed=11)).run().check()


@pytest.mark.parametrize("ratio", [1, 2, 3, 4, 8])
def test_head_ratios(ratio):
    """H_v = ratio * H_k: every CTA convolves its key head's q / k channels
    itself (v-head h reads key head h / ratio); the new conv slot's q / k
    channels are written by the key head's first v-head only."""
    case = _case(batch=5, H_k=2, H_v=2 * ratio, seed=90 + ratio)
    Step(case, synth.conv_inputs(case, seed=14 + ratio)).run().check()


@pytest.mark.parametrize("flags", [1, 3, 7])
def test_early_read_flags(flags):
    """The early-read flags (with 7 the conv history and the state tile are
    read before the dependency wait) give the oracle's results and the same
    bits as flags = 0."""
    case = _case(batch=8, seed=95, extra_rows=5, pad_prob=0.1)
    ci = synth.conv_inputs(case, seed=19)
    base = Step(case, ci).run()
    flagged = Step(case, ci).run(flags=flags).check()
    assert torch.equal(base.out.view(torch.int16), flagged.out.view(torch.int16))
    assert torch.equal(base.conv.view(torch.int16), flagged.conv.view(torch.int16))
    dt = torch.int32 if case.state_dtype == synth.F32 else torch.int16
    assert torch.equal(base.pool.view(dt), flagged.pool.view(dt))


def test_zero_history_and_skipped_conv_writes():
    case = _case(batch=8, seed=83)
    ci = synth.conv_inputs(case, seed=12)
    conv_in, conv_out = ci.conv_in.copy(), ci.conv_out.copy()
    conv_in[::3] = -1
    conv_out[1::3] = -1
    Step(case, ci).run(conv_in, conv_out).check()


def test_mixed_batch_gather_and_padding():
    case = _case(batch=8, seed=84, extra_rows=11, pad_prob=0.15)
    Step(case, synth.conv_inputs(case, seed=13)).run().check()


def test_two_steps_rewind_through_gpu_written_slots():
    """Step 2 rewinds into the conv and state slots step 1 wrote, with fresh
    acceptance counts; the oracle does the same two calls."""
    c1 = _case(batch=5, seed=85, q_lens=[8, 8, 8, 8, 8])
    ci1 = synth.conv_inputs(c1, seed=14)
    s1 = Step(c1, ci1).run().check()
    c2 = _case(batch=5, seed=86)
    # step 2 reads the state slots step 1 wrote: slot of token (acc-1) in step 1's rows
    c2.state_indices[:, :] = -1
    free = np.setdiff1d(np.arange(c1.num_slots), c1.state_indices.ravel())
    for i in range(c2.batch):
        a = int(c2.num_accepted[i])
        c2.state_indices[i, max(a - 1, 0)] = c1.state_indices[i, max(a - 1, 0)]
        for t in range(int(c2.q_lens()[i])):
            if t != max(a - 1, 0):
                c2.state_indices[i, t] = free[i * c2.spec_stride + t]
    ci2 = synth.conv_inputs(c2, seed=15)
    ci2.pool = s1.conv_host
    s2 = Step(c2, ci2, pool=s1.pool, conv_pool=s1.conv)
    s2.host = s1.host.copy()                      # the oracle continues from its own step-1 pool
    # reads step 1's write slots, writes the slots step 1 read
    s2.run(conv_in=ci1.conv_out, conv_out=ci1.conv_in).check()


def test_full_size_batch_sampled():
    """32 sequences of 8 draft tokens, H_k = 2, H_v = 16, bf16 state, W = 4."""
    case = synth.make_case(batch=32, H_k=2, H_v=16, T=8, state_dtype=synth.BF16, num_slots=2 * 32 * 8, seed=87)
    Step(case, synth.conv_inputs(case, seed=16)).run().check()


def test_bad_conv_slot_is_flagged_and_skipped():
    case = _case(batch=4, seed=88, q_lens=[3, 3, 3, 3])
    ci = synth.conv_inputs(case, seed=17)
    conv_in = ci.conv_in.copy()
    conv_in[2] = ci.pool.shape[0] + 5
    st = Step(case, ci)
    before = st.conv.clone()
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    out = torch.zeros((case.num_tokens, case.H_v, case.V), dtype=torch.bfloat16, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    gdn.gdn_spec_decode_conv(
        t_bf16(ci.x, DEV), t_bf16(ci.weight, DEV), t_bf16(ci.bias, DEV), st.conv, t(conv_in), t(ci.conv_out),
        t_bf16(case.a, DEV), t_bf16(case.b, DEV), t_bf16(case.z, DEV), t(case.A_log), t_bf16(case.dt_bias, DEV),
        t_bf16(case.norm_w, DEV), st.pool, t(case.state_indices), t(case.num_accepted), t(case.cu_seqlens), out,
        H_k=case.H_k, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & gdn.binding.GDN_FLAG_SLOT_RANGE
    assert torch.equal(st.conv[int(ci.conv_out[2])].view(torch.int16), before[int(ci.conv_out[2])].view(torch.int16))
    assert not torch.equal(st.conv[int(ci.conv_out[0])].view(torch.int16),
                           before[int(ci.conv_out[0])].view(torch.int16))

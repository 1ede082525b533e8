"""Pins for the oracle's prefill routine: it must be the same per-token step
as the decode path, routed over a whole prompt (PR #52191 report,
implementation steps 3-5: the chunked prefill kernel carries the state across
the prompt and writes it back; its tests split a prompt over two calls)."""
from __future__ import annotations

import numpy as np
import pytest

from gated_deltanet_linear_sm_gb300 import synth
from oracle import oracle as orc
from tests.util import initial_pool


def _prompt_case(L=(13, 7, 20), H_k=2, H_v=4, state_dtype=synth.F32, seed=40):
    return synth.make_case(batch=len(L), H_k=H_k, H_v=H_v, T=max(L), state_dtype=state_dtype,
                           num_slots=64, q_lens=list(L), acc=[1] * len(L), seed=seed)


def _arrays(c):
    return dict(q=c.q, k=c.k, v=c.v, a=c.a, b=c.b, z=c.z, A_log=c.A_log, dt_bias=c.dt_bias,
                norm_w=c.norm_w, scale=c.scale, eps=c.eps)


def test_prefill_equals_spec_step_with_only_the_last_slot_written():
    """A prompt of L tokens from slot s equals the speculative step over the
    same tokens whose read position lies past the drafts and whose slot table
    holds only the last position."""
    c = _prompt_case()
    B = c.batch
    L = c.q_lens()
    reads = np.array([3, 9, 17], np.int32)
    writes = np.array([30, 31, 32], np.int32)
    pool = initial_pool(c).astype(np.float64)
    pool[reads] = np.random.default_rng(0).normal(0, 0.1, pool[reads].shape)
    p1 = pool.copy()
    r1 = orc.prefill(**_arrays(c), pool=p1, state_dtype=orc.F64, cu_seqlens=c.cu_seqlens,
                     read_slots=reads, write_slots=writes)
    stride = int(L.max()) + 1
    idx = np.full((B, stride), -1, np.int32)
    for i in range(B):
        idx[i, L[i] - 1] = writes[i]
        idx[i, stride - 1] = reads[i]
    p2 = pool.copy()
    r2 = orc.spec_decode(**_arrays(c), pool=p2, state_dtype=orc.F64, state_indices=idx,
                         num_accepted=np.full(B, stride, np.int32), cu_seqlens=c.cu_seqlens)
    np.testing.assert_array_equal(r1["out_f64"], r2["out_f64"])
    np.testing.assert_array_equal(p1, p2)


def test_zero_initial_state_equals_a_zeroed_slot():
    c = _prompt_case(seed=41)
    pool = initial_pool(c)
    pool[50:53] = 0.0
    p1, p2 = pool.copy(), pool.copy()
    r1 = orc.prefill(**_arrays(c), pool=p1, state_dtype=orc.F32, cu_seqlens=c.cu_seqlens,
                     read_slots=np.array([-1, -1, -1], np.int32), write_slots=np.array([5, 6, 7], np.int32))
    r2 = orc.prefill(**_arrays(c), pool=p2, state_dtype=orc.F32, cu_seqlens=c.cu_seqlens,
                     read_slots=np.array([50, 51, 52], np.int32), write_slots=np.array([5, 6, 7], np.int32))
    np.testing.assert_array_equal(r1["out_f64"], r2["out_f64"])
    np.testing.assert_array_equal(p1, p2)


def test_one_token_prompt_in_place_equals_ordinary_decode():
    c = synth.make_case(batch=6, H_k=1, H_v=8, T=1, state_dtype=synth.BF16, num_slots=32, acc=[1] * 6, seed=42)
    slots = c.state_indices[:, 0].copy()
    pool = initial_pool(c)
    p1, p2 = pool.copy(), pool.copy()
    r1 = orc.prefill(**_arrays(c), pool=p1, state_dtype=orc.BF16, cu_seqlens=c.cu_seqlens,
                     read_slots=slots, write_slots=slots)
    r2 = orc.decode_nonspec(**_arrays(c), pool=p2, state_dtype=orc.BF16, slots=slots)
    np.testing.assert_array_equal(r1["out_bf16"], r2["out_bf16"])
    np.testing.assert_array_equal(p1, p2)


@pytest.mark.parametrize("cut", [1, 6, 12])
def test_prompt_split_over_two_calls(cut):
    """Running the first `cut` tokens, storing the state, and resuming from
    that slot gives bit-identical outputs and final state with an unrounded
    (FP64) pool."""
    c = _prompt_case(L=(13, 15, 20), seed=43)
    B = c.batch
    reads = np.array([3, 9, 17], np.int32)
    mids = np.array([40, 41, 42], np.int32)
    writes = np.array([30, 31, 32], np.int32)
    pool = initial_pool(c).astype(np.float64)
    pool[reads] = np.random.default_rng(1).normal(0, 0.1, pool[reads].shape)
    whole = pool.copy()
    rw = orc.prefill(**_arrays(c), pool=whole, state_dtype=orc.F64, cu_seqlens=c.cu_seqlens,
                     read_slots=reads, write_slots=writes)
    cu = c.cu_seqlens.astype(np.int64)
    first = np.concatenate([np.arange(cu[i], cu[i] + cut) for i in range(B)])
    second = np.concatenate([np.arange(cu[i] + cut, cu[i + 1]) for i in range(B)])

    def sub(rows):
        return dict(q=c.q[rows], k=c.k[rows], v=c.v[rows], a=c.a[rows], b=c.b[rows], z=c.z[rows],
                    A_log=c.A_log, dt_bias=c.dt_bias, norm_w=c.norm_w, scale=c.scale, eps=c.eps)

    split = pool.copy()
    cu1 = np.concatenate([[0], np.cumsum([cut] * B)]).astype(np.int32)
    cu2 = np.concatenate([[0], np.cumsum(np.diff(cu) - cut)]).astype(np.int32)
    r1 = orc.prefill(**sub(first), pool=split, state_dtype=orc.F64, cu_seqlens=cu1, read_slots=reads,
                     write_slots=mids)
    r2 = orc.prefill(**sub(second), pool=split, state_dtype=orc.F64, cu_seqlens=cu2, read_slots=mids,
                     write_slots=writes)
    np.testing.assert_array_equal(np.concatenate([r1["out_f64"], r2["out_f64"]])[np.argsort(
        np.concatenate([first, second]))], rw["out_f64"])
    np.testing.assert_array_equal(split[writes], whole[writes])


def test_prefill_contract():
    c = _prompt_case(seed=44)
    pool = initial_pool(c)
    with pytest.raises(orc.OracleError):
        orc.prefill(**_arrays(c), pool=pool, state_dtype=orc.F32, cu_seqlens=c.cu_seqlens,
                    read_slots=np.array([1, 2, 3], np.int32), write_slots=np.array([5, 5, 7], np.int32))
    with pytest.raises(orc.OracleError):
        orc.prefill(**_arrays(c), pool=pool, state_dtype=orc.F32, cu_seqlens=c.cu_seqlens,
                    read_slots=np.array([1, 7, 3], np.int32), write_slots=np.array([5, 6, 7], np.int32))

"""Pins for the oracle's short causal convolution with rewind in front of the
step (gdn_oracle_spec_decode_conv).  What the convolution reads and writes
follows the PR #46090 report (implementation step 2: the conv state is a wide
rolling buffer, sliced per token, convolved and written back) and the PR
#51674 report (implementation step 3: the speculative path runs
causal_conv1d_update with rewind before the post-conv decode kernel); the
readings taken where the pages print no formula are stated in the oracle's
header comment.

The pins do not reuse the oracle's arithmetic: the convolution is np.convolve
over the time-ordered inputs, and the step is the matrix-form NumPy statement
in tests/ref_numpy.py.
"""
from __future__ import annotations

import numpy as np
import pytest

from gated_deltanet_linear_sm_gb300 import synth
from oracle import oracle as orc
from tests import ref_numpy
from tests.util import bf16_values

KD = 16            # small heads: the pins run the full step in NumPy


def _case(T=3, acc=(2, 0, 3, 1), H_k=1, H_v=2, seed=60, sti_rows=0):
    c = synth.make_case(batch=len(acc), H_k=H_k, H_v=H_v, T=T, state_dtype=synth.F32, num_slots=64,
                        K=KD, V=KD, acc=list(acc), extra_rows=sti_rows, seed=seed)
    return c


def _pool64(case, seed=0):
    rng = np.random.default_rng([seed, 7])
    return rng.normal(0.0, 0.1, (case.num_slots, case.H_v, case.K, case.V))


def _run(case, ci, pool, conv_pool, **kw):
    return orc.spec_decode_conv(
        x=ci.x, conv_weight=ci.weight, conv_bias=ci.bias, conv_pool=conv_pool,
        conv_in=kw.get("conv_in", ci.conv_in), conv_out=kw.get("conv_out", ci.conv_out),
        H_k=case.H_k, K=case.K, a=case.a, b=case.b, z=case.z, A_log=case.A_log, dt_bias=case.dt_bias,
        norm_w=case.norm_w, pool=pool, state_dtype=orc.F64, state_indices=case.state_indices,
        num_accepted=kw.get("num_accepted", case.num_accepted), cu_seqlens=case.cu_seqlens,
        spec_token_indx=case.spec_token_indx, scale=case.scale, eps=case.eps)


def _scalar(bits):
    return float(bf16_values(np.array([bits], np.uint16))[0])


def _rows(case, i):
    cu = case.cu_seqlens
    n = np.arange(cu[i], cu[i + 1])
    return case.spec_token_indx[n] if case.spec_token_indx is not None else n


def _numpy_reference(case, ci, pool, conv_pool):
    """Expected out_f64 of every processed token, by brute force."""
    W, D = ci.width, ci.conv_dim
    QK = case.H_k * case.K
    w = bf16_values(ci.weight)
    bias = bf16_values(ci.bias) if ci.bias is not None else np.zeros(D)
    x = bf16_values(ci.x)
    out = {}
    for i in range(case.batch):
        rows = _rows(case, i)
        ql = len(rows)
        acc = int(case.num_accepted[i])
        rj = max(acc - 1, 0)
        rs = int(case.state_indices[i, rj])
        if ql == 0 or rs < 0:
            continue
        a_eff = max(acc, 1)
        hist = bf16_values(conv_pool[ci.conv_in[i], a_eff:a_eff + W - 1]) if ci.conv_in[i] >= 0 \
            else np.zeros((W - 1, D))
        u = np.concatenate([hist, x[rows]], 0)                        # [W-1+ql, D] in time order
        y = np.empty((ql, D))
        for ch in range(D):
            pre = np.convolve(u[:, ch], w[ch, ::-1], mode="valid") + bias[ch]
            y[:, ch] = pre / (1.0 + np.exp(-pre))
        q = y[:, :QK].reshape(ql, case.H_k, case.K)
        k = y[:, QK:2 * QK].reshape(ql, case.H_k, case.K)
        v = y[:, 2 * QK:].reshape(ql, case.H_v, case.V)
        group = case.H_v // case.H_k
        for h in range(case.H_v):
            S = pool[rs, h].copy()
            for t, r in enumerate(rows):
                S, o = ref_numpy.token_step(
                    S, q[t, h // group], k[t, h // group], v[t, h],
                    _scalar(case.a[r, h]), _scalar(case.b[r, h]),
                    float(case.A_log[h]), _scalar(case.dt_bias[h]), scale=case.scale)
                out[(int(r), h)] = ref_numpy.gated_rmsnorm(
                    o, bf16_values(case.z[r, h]), bf16_values(case.norm_w), case.eps)
    return out


@pytest.mark.parametrize("width,with_bias", [(4, True), (2, False), (3, True)])
def test_matches_numpy_brute_force(width, with_bias):
    case = _case()
    ci = synth.conv_inputs(case, width=width, with_bias=with_bias, seed=1)
    pool = _pool64(case)
    expect = _numpy_reference(case, ci, pool, ci.pool)
    res = _run(case, ci, pool.copy(), ci.pool.copy())
    assert expect
    for (r, h), o in expect.items():
        np.testing.assert_allclose(res["out_f64"][r, h], o, rtol=1e-10, atol=1e-12)


def test_gathered_rows_of_a_mixed_batch():
    """Projection rows come through spec_token_indx like every other input."""
    case = _case(seed=61, sti_rows=5)
    ci = synth.conv_inputs(case, seed=2)
    pool = _pool64(case, 1)
    expect = _numpy_reference(case, ci, pool, ci.pool)
    res = _run(case, ci, pool.copy(), ci.pool.copy())
    for (r, h), o in expect.items():
        np.testing.assert_allclose(res["out_f64"][r, h], o, rtol=1e-10, atol=1e-12)


def test_new_slot_holds_history_then_raw_inputs():
    case = _case(seed=62)
    ci = synth.conv_inputs(case, seed=3)
    before = ci.pool.copy()
    cp = ci.pool.copy()
    _run(case, ci, _pool64(case), cp)
    W = ci.width
    for i in range(case.batch):
        rows = _rows(case, i)
        a_eff = max(int(case.num_accepted[i]), 1)
        got = cp[ci.conv_out[i]]
        np.testing.assert_array_equal(got[:W - 1], before[ci.conv_in[i], a_eff:a_eff + W - 1])
        np.testing.assert_array_equal(got[W - 1:W - 1 + len(rows)], ci.x[rows])
        np.testing.assert_array_equal(got[W - 1 + len(rows):], before[ci.conv_out[i], W - 1 + len(rows):])
    untouched = np.setdiff1d(np.arange(cp.shape[0]), ci.conv_out)
    np.testing.assert_array_equal(cp[untouched], before[untouched])


@pytest.mark.parametrize("accepted", [1, 2, 3])
def test_rewind_equals_fresh_history(accepted):
    """Step 1 writes its conv slot; step 2 with `accepted` tokens kept reads it
    back.  The same step 2 from a slot that holds, at rows 1 .. W-1, the last
    W-1 inputs of (step 1's history, step 1's first `accepted` inputs) with
    acceptance 1 gives identical outputs."""
    W = 4
    c1 = _case(T=3, acc=(1,), seed=63)
    ci1 = synth.conv_inputs(c1, width=W, num_conv_slots=4, seed=4)
    cp = ci1.pool.copy()
    pool = _pool64(c1, 2)
    _run(c1, ci1, pool, cp, conv_in=np.array([0], np.int32), conv_out=np.array([1], np.int32))
    x1 = ci1.x[_rows(c1, 0)]
    hist = ci1.pool[0, 1:W]                                      # what step 1 read (acceptance 1)
    kept = np.concatenate([hist, x1[:accepted]], 0)[-(W - 1):]
    c2 = _case(T=3, acc=(accepted,), seed=64)
    ci2 = synth.conv_inputs(c2, width=W, num_conv_slots=4, seed=5)
    ci2.pool[:] = cp
    ci2.pool[2, 1:W] = kept
    p_a, p_b = _pool64(c2, 3), _pool64(c2, 3)
    ra = _run(c2, ci2, p_a, ci2.pool.copy(), conv_in=np.array([1], np.int32), conv_out=np.array([3], np.int32))
    # the same SSM read slot, now as column 0 with acceptance 1; unused write slots
    rs = int(c2.state_indices[0, max(accepted - 1, 0)])
    free = [s for s in range(c2.num_slots) if s not in set(c2.state_indices.ravel().tolist())]
    idx_b = np.array([[rs, free[0], free[1]]], np.int32)
    rb = orc.spec_decode_conv(
        x=ci2.x, conv_weight=ci2.weight, conv_bias=ci2.bias, conv_pool=ci2.pool.copy(),
        conv_in=np.array([2], np.int32), conv_out=np.array([3], np.int32), H_k=c2.H_k, K=c2.K, a=c2.a,
        b=c2.b, z=c2.z, A_log=c2.A_log, dt_bias=c2.dt_bias, norm_w=c2.norm_w, pool=p_b, state_dtype=orc.F64,
        state_indices=idx_b,
        num_accepted=np.array([1], np.int32), cu_seqlens=c2.cu_seqlens, scale=c2.scale, eps=c2.eps)
    rows = _rows(c2, 0)
    np.testing.assert_array_equal(ra["out_f64"][rows], rb["out_f64"][rows])


def test_negative_read_slot_is_zero_history():
    case = _case(seed=65)
    ci = synth.conv_inputs(case, seed=6)
    zeroed = ci.pool.copy()
    zeroed[ci.conv_in] = 0
    r1 = _run(case, ci, _pool64(case, 4), zeroed)
    r2 = _run(case, ci, _pool64(case, 4), ci.pool.copy(), conv_in=np.full(case.batch, -1, np.int32))
    np.testing.assert_array_equal(r1["out_f64"], r2["out_f64"])


def test_contract():
    case = _case(seed=66)
    ci = synth.conv_inputs(case, seed=7)
    with pytest.raises(orc.OracleError):                         # in place: read slot written
        _run(case, ci, _pool64(case), ci.pool.copy(), conv_out=ci.conv_in.copy())
    with pytest.raises(orc.OracleError):                         # two sequences write one slot
        out = ci.conv_out.copy()
        out[1] = out[0]
        _run(case, ci, _pool64(case), ci.pool.copy(), conv_out=out)
    with pytest.raises(orc.OracleError):                         # slot out of range
        out = ci.conv_out.copy()
        out[0] = ci.pool.shape[0]
        _run(case, ci, _pool64(case), ci.pool.copy(), conv_out=out)
    short = synth.ConvInputs(width=ci.width, state_len=ci.state_len - 1, x=ci.x, weight=ci.weight,
                             bias=ci.bias, pool=np.ascontiguousarray(ci.pool[:, :-1]), conv_in=ci.conv_in,
                             conv_out=ci.conv_out)
    with pytest.raises(orc.OracleError):                         # state_len < W - 1 + spec_stride
        _run(case, short, _pool64(case), short.pool.copy())

"""Pins for the FP64 oracle: each test checks it against something other than
itself -- IEEE format definitions and library conversions, closed forms of the
gated delta rule, invariants of the slot routing, and an independently written
NumPy twin of one token step.

Where a pin follows a statement of the vLLM PR report pages, the page and
section are named in the test's docstring.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

from gated_deltanet_linear_sm_gb300 import synth
from oracle import oracle as orc
from tests import ref_numpy
from tests.util import (as_bf16_exact, bf16_values, f16_values, initial_pool,
                        one_sequence, rel_l2, state_values)

K = V = 128
SCALE = 128 ** -0.5


# --------------------------------------------------------------------------
# number formats
# --------------------------------------------------------------------------

def test_bf16_rounding_matches_library_on_f32_inputs():
    """RNE double->bf16 equals torch's float32->bfloat16 on float32 inputs,
    including exact ties between bf16 neighbours."""
    rng = np.random.default_rng(1)
    x = rng.normal(0, 1, 200000).astype(np.float32) * np.float32(2.0) ** rng.integers(-140, 120, 200000).astype(np.float32)
    # exact midpoints between adjacent bf16 values: low half = 0x8000
    mids = (rng.integers(0, 1 << 16, 20000, dtype=np.uint32) << 16 | 0x8000).astype(np.uint32).view(np.float32)
    x = np.concatenate([x, mids[np.isfinite(mids)], np.array([0.0, -0.0, 3.4e38, -3.4e38, 1e-45], np.float32)])
    got = orc.round_bf16(x.astype(np.float64))
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)


def test_bf16_rounding_is_nearest_even_on_f64_inputs():
    """For doubles (not float32-exact), the bf16 result is at least as near as
    both bit-adjacent bf16 values, and an exact tie picks the even pattern."""
    rng = np.random.default_rng(2)
    x = rng.normal(0, 1, 50000) * 2.0 ** rng.integers(-130, 125, 50000)
    x = x[np.abs(x) < 3.3e38]
    bits = orc.round_bf16(x)
    y = bf16_values(bits)
    mag = bits & 0x7FFF
    sgn = bits & 0x8000
    up = bf16_values((sgn | np.minimum(mag + 1, 0x7F7F)).astype(np.uint16))
    dn = bf16_values((sgn | np.maximum(mag.astype(np.int64) - 1, 0)).astype(np.uint16))
    e = np.abs(x - y)
    assert np.all(e <= np.abs(x - up)) and np.all(e <= np.abs(x - dn))
    ties = (e == np.abs(x - up)) | (e == np.abs(x - dn))
    ties &= e > 0
    assert np.all(bits[ties] % 2 == 0)


def test_f16_rounding_matches_numpy():
    """RNE double->fp16, with gradual underflow and overflow, equals NumPy's
    float64->float16 conversion."""
    rng = np.random.default_rng(3)
    x = rng.normal(0, 1, 200000) * 2.0 ** rng.integers(-30, 18, 200000)
    # exact ties at subnormal and normal spacings, and the overflow edge
    ties = np.concatenate([(np.arange(1, 2000) + 0.5) * 2.0 ** -24,
                           (1024 + np.arange(0, 1023) + 0.5) * 2.0 ** -10,
                           [65504.0, 65519.99, 65520.0, 65536.0, 2.0 ** -25, 0.0]])
    x = np.concatenate([x, ties, -ties])
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(orc.round_f16(x), want)


def test_f32_rounding_matches_numpy():
    rng = np.random.default_rng(4)
    x = rng.normal(0, 1, 100000) * 2.0 ** rng.integers(-150, 128, 100000)
    with np.errstate(over="ignore"):
        want = x.astype(np.float32)
    got = orc.round_f32(x)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_bit_decoding_exhaustive():
    """Every one of the 65536 bf16 and fp16 patterns decodes to the library's value."""
    pats = np.arange(1 << 16, dtype=np.uint16)
    got = orc.value_bf16(pats)
    want = bf16_values(pats)
    same = (got == want) | (np.isnan(got) & np.isnan(want))
    assert same.all()
    got = orc.value_f16(pats)
    want = f16_values(pats)
    same = (got == want) | (np.isnan(got) & np.isnan(want))
    assert same.all()


# --------------------------------------------------------------------------
# closed forms of one step
# --------------------------------------------------------------------------

def _axis(m, c=256.0, n=K):
    e = np.zeros(n)
    e[m] = c
    return e


def _rand(rng, shape, s=1.0):
    return as_bf16_exact(rng.normal(0, s, shape))


def _khat_norm2(c=256.0):
    # |k^|^2 for k = c * e_m under the 1e-6 epsilon reading
    return c * c / (c * c + 1e-6)


def test_beta_half_scale_and_update_from_zero_state():
    """S0 = 0, b = 0 (beta = 1/2), k = q on one axis: the update writes
    beta * v into that key row and the readout is beta * scale * v.
    (PR #51674 report, implementation step 2: scale = 128^-0.5.)"""
    rng = np.random.default_rng(10)
    v = _rand(rng, V)
    r = one_sequence(np.zeros((K, V)), [dict(q=_axis(3), k=_axis(3), v=v, a=0.0, b=0.0)])
    kh = math.sqrt(_khat_norm2())
    np.testing.assert_allclose(r["out"][0], 0.5 * SCALE * v * kh * kh, rtol=1e-13, atol=1e-300)
    S1 = r["states"][0]
    np.testing.assert_allclose(S1[3], 0.5 * v * kh, rtol=1e-13)
    assert np.all(S1[np.arange(K) != 3] == 0.0)


@pytest.mark.parametrize("x", [-3.0, 0.0, 0.5, 4.0, 19.5, 25.0])
def test_decay_gate_closed_form(x):
    """beta ~ 0 (b = -88) leaves S1 = exp(g) S0, and with A_log = 0 the decay
    exp(-softplus(x)) equals 1 / (1 + e^x) for x below the softplus threshold
    and e^-x above it (reading: threshold 20)."""
    rng = np.random.default_rng(11)
    S0 = rng.normal(0, 0.1, (K, V))
    r = one_sequence(S0, [dict(q=_rand(rng, K), k=_rand(rng, K), v=_rand(rng, V), a=x, b=-88.0)])
    decay = 1.0 / (1.0 + math.exp(x)) if x <= 20 else math.exp(-x)
    np.testing.assert_allclose(r["states"][0], decay * S0, rtol=1e-12, atol=1e-30)


def test_decay_gate_scales_with_exp_A_log():
    """exp(g) = (1 + e^x)^(-exp(A_log)): A_log enters through its exponential."""
    rng = np.random.default_rng(12)
    S0 = rng.normal(0, 0.1, (K, V))
    A_log = float(np.float32(math.log(3.0)))
    x = 0.75
    r = one_sequence(S0, [dict(q=_rand(rng, K), k=_rand(rng, K), v=_rand(rng, V), a=x, b=-88.0)],
                     A_log=A_log)
    decay = (1.0 + math.exp(x)) ** (-math.exp(A_log))
    np.testing.assert_allclose(r["states"][0], decay * S0, rtol=1e-12)


def test_no_decay_when_A_log_is_minus_infinity():
    rng = np.random.default_rng(13)
    S0 = rng.normal(0, 0.1, (K, V))
    r = one_sequence(S0, [dict(q=_rand(rng, K), k=_rand(rng, K), v=_rand(rng, V), a=1.0, b=-88.0)],
                     A_log=-math.inf)
    np.testing.assert_allclose(r["states"][0], S0, rtol=1e-15, atol=1e-37)


def test_dt_bias_adds_to_a():
    """The decay depends on a + dt_bias only."""
    rng = np.random.default_rng(14)
    S0 = rng.normal(0, 0.1, (K, V))
    toks = dict(q=_rand(rng, K), k=_rand(rng, K), v=_rand(rng, V), b=-88.0)
    r1 = one_sequence(S0, [dict(toks, a=1.5)], dt_bias=-0.25)
    r2 = one_sequence(S0, [dict(toks, a=1.25)], dt_bias=0.0)
    np.testing.assert_array_equal(r1["states"], r2["states"])


@pytest.mark.parametrize("b", [88.0, 0.75, -1.5])
def test_delta_rule_closed_form(b):
    """After one token, S1^T k^ = (1 - beta |k^|^2) e^g S0^T k^ + beta |k^|^2 v;
    with beta = 1 this is the delta-rule overwrite S1^T k^ = v."""
    rng = np.random.default_rng(15)
    S0 = rng.normal(0, 0.1, (K, V))
    k = _rand(rng, K)
    v = _rand(rng, V)
    x = 0.3125                           # bf16-exact
    r = one_sequence(S0, [dict(q=_rand(rng, K), k=k, v=v, a=x, b=b)])
    beta = 1.0 / (1.0 + math.exp(-b))
    decay = 1.0 / (1.0 + math.exp(x))
    n2 = k @ k
    khat = k / math.sqrt(n2)             # unit key; the epsilon shifts |k^|^2 by ~1e-8
    lhs = r["states"][0].T @ khat
    rhs = (1 - beta) * decay * (S0.T @ khat) + beta * v
    np.testing.assert_allclose(lhs, rhs, rtol=1e-6, atol=1e-7)


def test_readout_is_transposed_state_times_query():
    """o = S^T q^: a one-hot query on key row m reads row m of the K x V state
    (not column m), times the scale."""
    rng = np.random.default_rng(16)
    S0 = rng.normal(0, 0.1, (K, V))
    m = 17
    r = one_sequence(S0, [dict(q=_axis(m), k=_rand(rng, K), v=_rand(rng, V), a=0.2, b=0.1)])
    S1 = r["states"][0]
    np.testing.assert_allclose(r["out"][0], SCALE * math.sqrt(_khat_norm2()) * S1[m], rtol=1e-12)
    assert rel_l2(r["out"][0], SCALE * S1[:, m]) > 0.5


def test_orthonormal_keys_multi_token_closed_form():
    """Keys on distinct axes: token t scales every row by e^{g_t} and replaces
    row p_t by (1 - beta_t) e^{g_t} S[p_t] + beta_t v_t.  Pins the serial token
    order and the per-token state writes (PR #46090 report, implementation
    step 3: each token's state goes to its own slot)."""
    rng = np.random.default_rng(17)
    S0 = rng.normal(0, 0.1, (K, V))
    T = 6
    rows = [5, 90, 5, 33, 127, 0]
    xs = [0.5, -1.0, 2.0, 0.0, -0.5, 1.25]
    bs = [0.25, -0.5, 1.0, 3.0, 0.0, -2.0]
    toks = [dict(q=_rand(rng, K), k=_axis(p), v=_rand(rng, V), a=x, b=b)
            for p, x, b in zip(rows, xs, bs)]
    r = one_sequence(S0, toks, state_dtype=orc.F32)
    S = S0.astype(np.float32).astype(np.float64)
    n2 = _khat_norm2()
    for t in range(T):
        decay = 1.0 / (1.0 + math.exp(xs[t]))
        beta = 1.0 / (1.0 + math.exp(-bs[t]))
        S = decay * S
        p = rows[t]
        S[p] = (1 - beta * n2) * S[p] + beta * math.sqrt(n2) * toks[t]["v"]
        np.testing.assert_allclose(r["states"][t], S, rtol=1e-12, atol=1e-300)
        # the slot written after token t holds the float32 rounding of S
        np.testing.assert_array_equal(r["pool"][t + 1, 0], S.astype(np.float32))


def test_rmsnorm_epilogue_closed_form():
    """With S0 = 0, one axis-aligned token and a constant v, o is the same in
    every column, so rmsnorm(o) = o / sqrt(o^2 + eps); silu(0) = 0 and
    silu(40) = 40 to double precision.  (PR #51674 report, implementation
    step 1: gated RMSNorm epilogue; step 2: norm_eps = 1e-5.)"""
    rng = np.random.default_rng(18)
    c = 0.75
    z = np.where(np.arange(V) % 2 == 0, 0.0, 40.0)
    w = _rand(rng, V, 0.1) + 1.0
    w = as_bf16_exact(w)
    r = one_sequence(np.zeros((K, V)), [dict(q=_axis(2), k=_axis(2), v=np.full(V, c), a=0.0, b=0.0, z=z)],
                     norm_w=w)
    o = 0.5 * SCALE * c * _khat_norm2()
    want = o / math.sqrt(o * o + 1e-5) * w * z
    np.testing.assert_allclose(r["out"][0], want, rtol=1e-13, atol=1e-300)


def test_silu_gate_odd_identity():
    """silu(-z) = silu(z) - z, so y(z) - y(-z) = rmsnorm(o) * w * z exactly in
    the outputs of two runs that differ only in the sign of z."""
    rng = np.random.default_rng(19)
    S0 = rng.normal(0, 0.1, (K, V))
    tok = dict(q=_rand(rng, K), k=_rand(rng, K), v=_rand(rng, V), a=0.1, b=0.2)
    z = _rand(rng, V, 2.0)
    w = as_bf16_exact(rng.normal(1, 0.1, V))
    rp = one_sequence(S0, [dict(tok, z=z)], norm_w=w)
    rm = one_sequence(S0, [dict(tok, z=-z)], norm_w=w)
    raw = one_sequence(S0, [tok])["out"][0]
    normed = raw / math.sqrt(np.mean(raw * raw) + 1e-5)
    np.testing.assert_allclose(rp["out"][0] - rm["out"][0], normed * w * z, rtol=1e-10, atol=1e-13)


def test_query_and_key_are_l2_normalised():
    """Scaling q and k by powers of two (exact in bf16) changes nothing beyond
    the epsilon's effect: q and k enter only through their directions."""
    rng = np.random.default_rng(20)
    S0 = rng.normal(0, 0.1, (K, V))
    q, k, v = _rand(rng, K), _rand(rng, K), _rand(rng, V)
    r1 = one_sequence(S0, [dict(q=q, k=k, v=v, a=0.3, b=0.4)])
    r2 = one_sequence(S0, [dict(q=4.0 * q, k=0.5 * k, v=v, a=0.3, b=0.4)])
    np.testing.assert_allclose(r2["out"], r1["out"], rtol=1e-7, atol=1e-9)
    np.testing.assert_allclose(r2["states"], r1["states"], rtol=1e-7, atol=1e-8)


def test_numpy_twin_single_token():
    """The C oracle's token step agrees with the independently written NumPy
    matrix-form twin, gated and ungated, to FP64 rounding."""
    rng = np.random.default_rng(21)
    S0 = rng.normal(0, 0.1, (K, V))
    q, k, v, z = _rand(rng, K), _rand(rng, K), _rand(rng, V), _rand(rng, V)
    w = as_bf16_exact(rng.normal(1, 0.1, V))
    a, b, dt = 0.625, -0.375, 0.5
    A_log = float(np.float32(math.log(5.0)))
    r = one_sequence(S0, [dict(q=q, k=k, v=v, a=a, b=b, z=z)], A_log=A_log, dt_bias=dt, norm_w=w)
    S1, o = ref_numpy.token_step(S0, q, k, v, a, b, A_log, dt, scale=SCALE)
    np.testing.assert_allclose(r["states"][0], S1, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(r["out"][0], ref_numpy.gated_rmsnorm(o, z, w, 1e-5), rtol=1e-11, atol=1e-14)


# --------------------------------------------------------------------------
# slot routing, composition, identities
# --------------------------------------------------------------------------

def _case_arrays(case):
    return dict(q=case.q, k=case.k, v=case.v, a=case.a, b=case.b, z=case.z, A_log=case.A_log,
                dt_bias=case.dt_bias, norm_w=case.norm_w, scale=case.scale, eps=case.eps)


def test_composition_of_single_token_calls():
    """A T-token call equals T chained one-token calls (num_accepted = 1, each
    reading the slot the previous call wrote), bit for bit, with an unrounded
    (FP64) pool.  Pins the rewind and the per-token slot routing."""
    case = synth.make_case(batch=3, H_k=1, H_v=2, T=4, state_dtype=synth.F32, num_slots=64,
                           acc=[1, 3, 4], seed=5)
    pool0 = initial_pool(case).astype(np.float64)
    poolA = pool0.copy()
    full = orc.spec_decode(**_case_arrays(case), pool=poolA, state_dtype=orc.F64,
                           state_indices=case.state_indices, num_accepted=case.num_accepted,
                           cu_seqlens=case.cu_seqlens)
    poolB = pool0.copy()
    for i in range(case.batch):
        acc = int(case.num_accepted[i])
        src = int(case.state_indices[i, max(acc - 1, 0)])
        for t in range(4):
            r = int(case.cu_seqlens[i]) + t
            dst = int(case.state_indices[i, t])
            # one token: write slot dst (position 0), read slot src (position acc-1 = 1)
            one = orc.spec_decode(
                q=case.q[r:r + 1], k=case.k[r:r + 1], v=case.v[r:r + 1], a=case.a[r:r + 1],
                b=case.b[r:r + 1], z=case.z[r:r + 1], A_log=case.A_log, dt_bias=case.dt_bias,
                norm_w=case.norm_w, pool=poolB, state_dtype=orc.F64,
                state_indices=np.array([[dst, src]], np.int32),
                num_accepted=np.array([2], np.int32), cu_seqlens=np.array([0, 1], np.int32))
            np.testing.assert_array_equal(one["out_f64"][0], full["out_f64"][r])
            src = dst
    # the read slot of each sequence is also written at t = acc-1; compare all slots
    np.testing.assert_array_equal(poolA, poolB)


def test_T1_accepted1_equals_ordinary_decode():
    """T = 1 with num_accepted = 1 reads and writes state_indices[i, 0] in
    place: ordinary recurrent decode (PR #51812 report, key source snippet:
    the non-spec update with ssm_state_indices)."""
    case = synth.make_case(batch=5, H_k=1, H_v=8, T=1, state_dtype=synth.F32, num_slots=16,
                           acc=[1] * 5, seed=6)
    pool_spec = initial_pool(case)
    pool_dec = pool_spec.copy()
    r1 = orc.run_case(case, pool_spec)
    r2 = orc.decode_nonspec(**{k: v for k, v in _case_arrays(case).items()}, pool=pool_dec,
                            state_dtype=orc.F32, slots=case.state_indices[:, 0].copy())
    np.testing.assert_array_equal(r1["out_bf16"], r2["out_bf16"])
    np.testing.assert_array_equal(r1["out_f64"], r2["out_f64"])
    np.testing.assert_array_equal(pool_spec, pool_dec)


def test_num_accepted_zero_clamps_to_first_slot():
    """num_accepted = 0 reads state_indices[i, 0], like num_accepted = 1, and
    never position -1 (PR #46090 report, review highlights: the acc-1
    underflow fix).  A guard entry in front of the index table points at a
    NaN-filled slot; reading it would poison every output."""
    case = synth.make_case(batch=2, H_k=1, H_v=2, T=3, state_dtype=synth.F32, num_slots=16,
                           acc=[0, 2], seed=7)
    pool = initial_pool(case)
    guard_slot = int(np.setdiff1d(np.arange(16), case.state_indices.ravel())[0])
    pool[guard_slot] = np.nan
    buf = np.concatenate([[guard_slot], case.state_indices.ravel()]).astype(np.int32)
    idx_view = buf[1:].reshape(case.state_indices.shape)
    p0 = pool.copy()
    r0 = orc.spec_decode(**_case_arrays(case), pool=p0, state_dtype=orc.F32, state_indices=idx_view,
                         num_accepted=np.array([0, 2], np.int32), cu_seqlens=case.cu_seqlens)
    p1 = pool.copy()
    r1 = orc.spec_decode(**_case_arrays(case), pool=p1, state_dtype=orc.F32,
                         state_indices=case.state_indices,
                         num_accepted=np.array([1, 2], np.int32), cu_seqlens=case.cu_seqlens)
    assert np.isfinite(r0["out_f64"]).all()
    np.testing.assert_array_equal(r0["out_f64"], r1["out_f64"])
    np.testing.assert_array_equal(p0, p1)


def test_slot_invariants_and_padding():
    """Untouched slots stay bit-identical, every valid write slot is written
    (NaN sentinels become finite), padded (-1) write slots are skipped, a
    padded read slot skips the whole sequence and its out rows, and q_len = 0
    sequences are skipped.  (PR #51674 report, review highlights: the kernel
    writes only unpadded rows.)"""
    case = synth.make_case(batch=12, H_k=1, H_v=4, T=4, state_dtype=synth.F32, num_slots=200,
                           q_lens=[4, 4, 0, 3, 4, 1, 4, 4, 2, 4, 4, 4],
                           acc=[0, 1, 2, 3, 4, 1, 2, 3, 1, 4, 2, 1], seed=8)
    idx = case.state_indices
    idx[1, 2] = -1                                   # padded write slot
    idx[6, 1] = -1                                   # padded read slot (acc = 2): sequence skipped
    pool = initial_pool(case)
    background = np.random.default_rng(0).normal(0, 1, pool.shape).astype(np.float32)
    untouched = np.ones(case.num_slots, bool)
    ql = case.q_lens()
    reads = case.read_slots()
    written = set()
    for i in range(case.batch):
        if ql[i] <= 0 or reads[i] < 0:
            continue
        for t in range(ql[i]):
            if idx[i, t] >= 0:
                written.add(int(idx[i, t]))
    read_set = {int(s) for s in reads if s >= 0}
    for s in range(case.num_slots):
        if s in written or s in read_set:
            untouched[s] = False
    pool[untouched] = background[untouched]
    write_only = sorted(written - read_set)
    pool[write_only] = np.nan
    before = pool.copy()
    res = orc.run_case(case, pool)
    assert np.array_equal(pool[untouched].view(np.uint32), before[untouched].view(np.uint32))
    assert np.isfinite(pool[sorted(written)]).all()
    # the slots of skipped sequences (q_len = 0, or a padded read slot) are untouched
    for i in (2, 6):
        for s in idx[i]:
            if s >= 0 and int(s) not in written:
                assert np.array_equal(pool[s].view(np.uint32), before[s].view(np.uint32))
    rows_active = set()
    for i in range(case.batch):
        if ql[i] > 0 and reads[i] >= 0:
            rows_active.update(range(int(case.cu_seqlens[i]), int(case.cu_seqlens[i + 1])))
    for r in range(case.num_tokens):
        assert np.isnan(res["out_f64"][r]).all() == (r not in rows_active)


def _gathered_case():
    return synth.make_case(batch=6, H_k=2, H_v=16, T=3, state_dtype=synth.F16, num_slots=64,
                           extra_rows=9, seed=9)


def test_mixed_batch_gather_equals_pre_gathered_rows():
    """Gathering q/k/v/a/b/z through spec_token_indx gives bit-identical
    results to passing the gathered rows directly, and writes out only at the
    gathered rows (PR #51812 report, implementation steps 2-3)."""
    case = _gathered_case()
    rows = case.spec_token_indx.astype(np.int64)
    pool_g = initial_pool(case)
    pool_d = pool_g.copy()
    rg = orc.run_case(case, pool_g)
    rd = orc.spec_decode(
        q=case.q[rows], k=case.k[rows], v=case.v[rows], a=case.a[rows], b=case.b[rows],
        z=case.z[rows], A_log=case.A_log, dt_bias=case.dt_bias, norm_w=case.norm_w, pool=pool_d,
        state_dtype=case.state_dtype, state_indices=case.state_indices,
        num_accepted=case.num_accepted, cu_seqlens=case.cu_seqlens)
    np.testing.assert_array_equal(rg["out_bf16"][rows], rd["out_bf16"])
    np.testing.assert_array_equal(pool_g, pool_d)
    others = np.setdiff1d(np.arange(case.num_tokens), rows)
    assert np.isnan(rg["out_f64"][others]).all()


def test_gate_misalignment_bug_would_be_caught():
    """Plant the bug the PR #51812 report fixes (q/k/v gathered, a/b consumed
    as the first T_spec rows) in the oracle's inputs: the outputs then differ
    from the aligned ones, so the gather test above detects that class."""
    case = _gathered_case()
    rows = case.spec_token_indx.astype(np.int64)
    n = len(rows)
    pool_ok = initial_pool(case)
    pool_bug = pool_ok.copy()
    ok = orc.spec_decode(
        q=case.q[rows], k=case.k[rows], v=case.v[rows], a=case.a[rows], b=case.b[rows],
        z=case.z[rows], A_log=case.A_log, dt_bias=case.dt_bias, norm_w=case.norm_w, pool=pool_ok,
        state_dtype=case.state_dtype, state_indices=case.state_indices,
        num_accepted=case.num_accepted, cu_seqlens=case.cu_seqlens)
    bug = orc.spec_decode(
        q=case.q[rows], k=case.k[rows], v=case.v[rows], a=case.a[:n], b=case.b[:n],
        z=case.z[rows], A_log=case.A_log, dt_bias=case.dt_bias, norm_w=case.norm_w, pool=pool_bug,
        state_dtype=case.state_dtype, state_indices=case.state_indices,
        num_accepted=case.num_accepted, cu_seqlens=case.cu_seqlens)
    assert rel_l2(bug["out_f64"], ok["out_f64"]) > 1e-2


def test_gqa_head_map_is_not_interleaved():
    """v-head h uses k-head h / (H_v / H_k) (PR #46090 report, fla.cpp
    listing): with H_k = 2, H_v = 16, heads 0-7 match an H_k = 1 run on k-head
    0's q/k and heads 8-15 one on k-head 1's."""
    case = synth.make_case(batch=3, H_k=2, H_v=16, T=2, state_dtype=synth.F32, num_slots=32, seed=10)
    pool = initial_pool(case)
    full = orc.run_case(case, pool.copy())
    for kh in range(2):
        heads = slice(8 * kh, 8 * kh + 8)
        sub_pool = np.ascontiguousarray(pool[:, heads])
        r = orc.spec_decode(
            q=case.q[:, kh:kh + 1], k=case.k[:, kh:kh + 1], v=case.v[:, heads], a=case.a[:, heads],
            b=case.b[:, heads], z=case.z[:, heads], A_log=case.A_log[heads],
            dt_bias=case.dt_bias[heads], norm_w=case.norm_w, pool=sub_pool, state_dtype=orc.F32,
            state_indices=case.state_indices, num_accepted=case.num_accepted,
            cu_seqlens=case.cu_seqlens)
        np.testing.assert_array_equal(r["out_f64"], full["out_f64"][:, heads])


def test_narrow_state_write_rounds_once_from_wide_carry():
    """With a bf16 / fp16 pool, each written slot is the RNE rounding of the
    FP64 carried state, which itself is never rounded (PR #52191 report,
    implementation step 4: compute wide, store narrow)."""
    for sd in (synth.BF16, synth.F16):
        case = synth.make_case(batch=4, H_k=1, H_v=2, T=4, state_dtype=sd, num_slots=32,
                               acc=[4, 4, 4, 4], seed=11)
        pool = initial_pool(case)
        res = orc.run_case(case, pool, states_T=4)
        rnd = orc.round_bf16 if sd == synth.BF16 else orc.round_f16
        for i in range(case.batch):
            for t in range(4):
                s = case.state_indices[i, t]
                np.testing.assert_array_equal(pool[s], rnd(res["states"][i, :, t]))
        # the carry is not re-rounded: the FP64 state after the last token is
        # not on the narrow grid
        vals = state_values(rnd(res["states"][:, :, 3]), sd)
        assert np.any(vals != res["states"][:, :, 3])


def test_contract_violations_are_rejected():
    case = synth.make_case(batch=3, H_k=1, H_v=2, T=2, state_dtype=synth.F32, num_slots=16,
                           acc=[1, 2, 1], seed=12)
    base = initial_pool(case)
    kw = _case_arrays(case)

    def run(**over):
        args = dict(state_indices=case.state_indices, num_accepted=case.num_accepted,
                    cu_seqlens=case.cu_seqlens)
        args.update(over)
        return orc.spec_decode(**kw, pool=base.copy(), state_dtype=orc.F32, **args)

    run()
    with pytest.raises(orc.OracleError, match="num_accepted"):
        run(num_accepted=np.array([3, 1, 1], np.int32))
    dup = case.state_indices.copy()
    dup[1, 1] = dup[0, 0]
    with pytest.raises(orc.OracleError, match="shared"):
        run(state_indices=dup)
    big = case.state_indices.copy()
    big[2, 1] = 16
    with pytest.raises(orc.OracleError, match="num_slots"):
        run(state_indices=big)
    with pytest.raises(orc.OracleError, match="q_len"):
        run(cu_seqlens=np.array([0, 3, 4, 6], np.int32))

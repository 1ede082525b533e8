"""Seeded randomised configurations against the oracle: the decode step over
batch sizes, head ratios, draft depths, acceptance and padding patterns,
gathered rows, state dtypes and every split code; the chunked prefill over
prompt-length mixes, head ratios and state dtypes; and the fused-conv step
over widths, bias, head ratios, lengths, padding, gathers and flags.  Each configuration is
drawn from a fixed seed, so a failure names a reproducible case."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import gated_deltanet_linear_sm_gb300 as gdn
from gated_deltanet_linear_sm_gb300 import synth
from tests.test_gpu_parity import _full_check
from tests.test_gpu_prefill import _case, _check, _run, _slots

pytestmark = pytest.mark.gpu

SPLITS = (0, 1, 2, 4, 8, 0x102, 0x104, 0x201, 0x202)
DTYPES = (synth.F32, synth.BF16, synth.F16)


def _decode_config(seed):
    rng = np.random.default_rng(1000 + seed)
    H_k = int(rng.choice([1, 2, 3, 4]))
    ratio = int(rng.choice([1, 2, 4, 8]))
    T = int(rng.integers(1, 9))
    batch = int(rng.integers(1, 41))
    sd = int(rng.choice(DTYPES))
    split = int(rng.choice(SPLITS))
    stride = T + int(rng.integers(0, 3)) if T < 8 else 8
    return dict(batch=batch, H_k=H_k, H_v=H_k * ratio, T=T, state_dtype=sd,
                num_slots=int(max(64, batch * stride + 16)), spec_stride=stride,
                q_lens=rng.choice([None, "ragged"]), acc=str(rng.choice(["uniform", "binomial"])),
                pad_prob=float(rng.choice([0.0, 0.1, 0.3])), extra_rows=int(rng.choice([0, 0, 17])),
                gated=bool(rng.random() > 0.2), seed=2000 + seed), split


@pytest.mark.parametrize("seed", range(64))
def test_decode_random_configuration(cuda_device, seed):
    """One random decode configuration (see _decode_config), every sequence
    compared with the oracle; the bound depends on the state dtype only."""
    kw, split = _decode_config(seed)
    case = synth.make_case(**kw)
    m = _full_check(case, cuda_device, split)
    assert m["out_rel_l2"] < 5e-4


def _prefill_config(seed):
    rng = np.random.default_rng(3000 + seed)
    H_k = int(rng.choice([1, 2, 3]))
    ratio = int(rng.choice([1, 2, 4, 8]))
    n = int(rng.integers(1, 13))
    lens = [int(x) for x in rng.choice([0, 1, 5, 63, 64, 65, 127, 128, 129, 200, 300], size=n)]
    if max(lens) == 0:
        lens[0] = 17
    sd = int(rng.choice(DTYPES))
    return lens, sd, H_k, H_k * ratio, bool(rng.random() > 0.2), 4000 + seed


@pytest.mark.parametrize("seed", range(24))
def test_chunked_prefill_random_configuration(seed):
    """One random prefill configuration (prompt lengths around the 64-token
    chunk boundaries, empty prompts, head ratios, gated or not, zero or slot
    initial states, skipped final writes), both prefill entry points against
    the oracle."""
    lens, sd, H_k, H_v, gated, s = _prefill_config(seed)
    case = synth.make_case(batch=len(lens), H_k=H_k, H_v=H_v, T=max(lens), state_dtype=sd,
                           num_slots=max(4 * len(lens) + 8, 32), spec_stride=1, q_lens=lens, acc=[1] * len(lens),
                           gated=gated, seed=s)
    reads, writes = _slots(case, s)
    for entry in ("chunked", "recurrent"):
        _check(entry, case, *_run(entry, case, reads, writes), writes)


def _conv_config(seed):
    rng = np.random.default_rng(5000 + seed)
    H_k = int(rng.choice([1, 2, 3]))
    ratio = int(rng.choice([1, 2, 3, 4, 8]))
    T = int(rng.integers(1, 9))
    batch = int(rng.integers(1, 25))
    return dict(batch=batch, H_k=H_k, H_v=H_k * ratio, T=T, state_dtype=int(rng.choice(DTYPES)),
                num_slots=2 * batch * T + 8, q_lens=rng.choice([None, "ragged"]),
                pad_prob=float(rng.choice([0.0, 0.1])), extra_rows=int(rng.choice([0, 0, 9])),
                seed=6000 + seed), int(rng.integers(1, 5)), bool(rng.random() > 0.3), int(rng.choice([0, 1, 3, 7]))


@pytest.mark.parametrize("seed", range(24))
def test_conv_random_configuration(seed):
    """One random fused-conv step (width 1-4, bias or none, head ratios,
    draft depth, ragged lengths, padded slots, gathered rows, state dtype,
    early-read flags) against the oracle; the new conv slots bit for bit."""
    from tests.gpu_util import active_rows
    from tests.test_gpu_conv import Step
    kw, width, bias, flags = _conv_config(seed)
    case = synth.make_case(**kw)
    if not len(active_rows(case)):                     # nothing to compare: every sequence skipped
        kw.update(q_lens=None, pad_prob=0.0)
        case = synth.make_case(**kw)
    ci = synth.conv_inputs(case, width=width, with_bias=bias, seed=7000 + seed)
    Step(case, ci).run(flags=flags).check()

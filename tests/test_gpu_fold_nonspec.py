"""Non-speculative decode tokens folded into the same launch as the
speculative sequences.

A mixed batch (PR #51812 report, motivation: non-spec tokens placed among
spec tokens) used to need two kernels: the spec step over the rows gathered by
spec_token_indx, and ordinary in-place decode over the rest (PR #51812 report,
key source snippet: the non-spec update with ssm_state_indices).  The PR
#51674 report's "evolution trade-offs" note records that the fused path gave
up mixed-batch fusion.  With this ABI a non-spec token is just a sequence with
q_len = 1, num_accepted = 1 and slot row [slot, -1, ...]: it reads and writes
its slot in place.  One launch then covers the whole mixed batch; the oracle
checks the spec part with its spec step and the folded part with its separate
ordinary-decode routine.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import gated_deltanet_linear_sm_gb300 as gdn
from gated_deltanet_linear_sm_gb300 import synth
from oracle import oracle as orc
from tests.gpu_util import device_tensors, make_pool, to_host_bits
from tests.util import bf16_values, rel_l2, state_values

pytestmark = pytest.mark.gpu


def fold(case, nonspec_rows, nonspec_slots):
    """Metadata for one launch: the case's spec sequences followed by one
    q_len = 1 sequence per non-spec token (host-side integer bookkeeping)."""
    B, S = case.state_indices.shape
    n = len(nonspec_rows)
    idx = np.full((B + n, S), -1, dtype=np.int32)
    idx[:B] = case.state_indices
    idx[B:, 0] = nonspec_slots
    acc = np.concatenate([case.num_accepted, np.ones(n, np.int32)]).astype(np.int32)
    cu = np.concatenate([case.cu_seqlens, case.cu_seqlens[-1] + 1 + np.arange(n)]).astype(np.int32)
    rows = np.concatenate([case.spec_token_indx, nonspec_rows]).astype(np.int32)
    return idx, acc, cu, rows


@pytest.mark.parametrize("split", [0, 1, 8])
def test_mixed_batch_in_one_launch(split):
    dev = torch.device("cuda", 0)
    case = synth.mixed(0)                                    # 48 spec seqs T=3 among 224 rows, fp16 state
    nonspec_rows = np.setdiff1d(np.arange(case.num_tokens), case.spec_token_indx).astype(np.int32)
    used = set(int(s) for s in case.state_indices.ravel() if s >= 0)
    free = np.array(sorted(set(range(case.num_slots)) - used))
    rng = np.random.default_rng(5)
    nonspec_slots = rng.choice(free, len(nonspec_rows), replace=False).astype(np.int32)
    idx, acc, cu, rows = fold(case, nonspec_rows, nonspec_slots)

    pool = make_pool(case, dev, slots=np.concatenate([case.touched_slots(), nonspec_slots]))
    host_pool = to_host_bits(pool)
    t = device_tensors(case, dev)
    out = torch.zeros(case.num_tokens, case.H_v, case.V, dtype=torch.bfloat16, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    gdn.gdn_spec_decode(t["q"], t["k"], t["v"], t["a"], t["b"], t["z"], t["A_log"], t["dt_bias"], t["norm_w"],
                        pool, torch.from_numpy(idx).to(dev), torch.from_numpy(acc).to(dev),
                        torch.from_numpy(cu).to(dev), out, spec_token_indx=torch.from_numpy(rows).to(dev),
                        max_T=3, split=split, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0

    # oracle: spec step over the gathered rows, ordinary decode over the others
    hp = host_pool.copy()
    spec = orc.run_case(case, hp)
    ns = orc.decode_nonspec(q=case.q[nonspec_rows], k=case.k[nonspec_rows], v=case.v[nonspec_rows],
                            a=case.a[nonspec_rows], b=case.b[nonspec_rows], z=case.z[nonspec_rows],
                            A_log=case.A_log, dt_bias=case.dt_bias, norm_w=case.norm_w, pool=hp,
                            state_dtype=case.state_dtype, slots=nonspec_slots)
    want = spec["out_bf16"].copy()
    want[nonspec_rows] = ns["out_bf16"]
    # rows of padded spec sequences are written by neither side
    act = np.isfinite(spec["out_f64"][:, 0, 0])
    act[nonspec_rows] = True
    got = bf16_values(out.view(torch.int16).cpu().numpy().view(np.uint16))
    assert rel_l2(got[act], bf16_values(want[act])) < 5e-4
    # every slot either path wrote
    gp = state_values(to_host_bits(pool), case.state_dtype)
    wp = state_values(hp, case.state_dtype)
    assert np.all(np.abs(gp - wp) <= 3e-2 + 3e-2 * np.abs(wp))
    changed = np.any(hp.reshape(case.num_slots, -1) != host_pool.reshape(case.num_slots, -1), axis=1)
    assert changed[nonspec_slots].all()

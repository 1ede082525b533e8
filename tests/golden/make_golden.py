"""Writes tests/golden/tiny_oracle.json: sampled FP64 oracle results on the
tiny workload (2 sequences, H_k=1, H_v=8, T=2, acceptance [1, 2], fp32 pool of
8 slots, seed 0).  Calls only the oracle (inputs come from the seeded
generator).  Re-run only when the oracle's arithmetic changes for a reason
named in the commit message.

    python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from gated_deltanet_linear_sm_gb300 import synth  # noqa: E402
from oracle import oracle as orc  # noqa: E402

STEP = 37


def compute():
    case = synth.tiny(0)
    pool = np.zeros((case.num_slots, case.H_v, case.K, case.V), np.float32)
    touched = case.touched_slots()
    pool[touched] = case.slot_values(touched)
    res = orc.run_case(case, pool, states_T=2)
    out = res["out_f64"].ravel()
    states = res["states"].ravel()
    written = sorted({int(s) for s in case.state_indices.ravel() if s >= 0})
    return {
        "workload": "tiny: B=2, H_k=1, H_v=8, K=V=128, T=2, num_accepted=[1,2], fp32 pool of 8 slots, seed 0",
        "state_indices": case.state_indices.tolist(),
        "out_sample_step": STEP,
        "out_sample": [float(x).hex() for x in out[::STEP]],
        "states_sample": [float(x).hex() for x in states[::STEP * 97]],
        "out_bf16_sum": int(res["out_bf16"].astype(np.int64).sum()),
        "pool_written_f32_sum": float(pool[written].astype(np.float64).sum()).hex(),
    }


if __name__ == "__main__":
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_oracle.json")
    with open(path, "w") as f:
        json.dump(compute(), f, indent=1)
    print("wrote", path)

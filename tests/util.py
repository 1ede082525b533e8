"""Small helpers shared by the tests: bf16 conversions (library routines),
explicit hand-built problems for the oracle pins, and comparison metrics."""
from __future__ import annotations

import numpy as np
import torch

from oracle import oracle as orc


def bf16_bits(x) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def bf16_values(bits) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)
    return torch.from_numpy(b.copy()).view(torch.bfloat16).to(torch.float64).numpy()


def f16_values(bits) -> np.ndarray:
    return np.ascontiguousarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def as_bf16_exact(x) -> np.ndarray:
    """Values of x after rounding to bf16, as float64."""
    return bf16_values(bf16_bits(x))


def state_values(pool, state_dtype) -> np.ndarray:
    if state_dtype == orc.F32:
        return pool.astype(np.float64)
    if state_dtype == orc.BF16:
        return bf16_values(pool)
    if state_dtype == orc.F16:
        return f16_values(pool)
    return pool.astype(np.float64)


def rel_l2(x, ref) -> float:
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref.ravel())
    return float(np.linalg.norm((x - ref).ravel()) / (den if den > 0 else 1.0))


def one_sequence(S0, tokens, *, A_log=0.0, dt_bias=0.0, norm_w=None, acc=1,
                 state_dtype=orc.F64, scale=128 ** -0.5, eps=1e-5, num_threads=1):
    """Run the oracle on one sequence with H_k = H_v = 1.

    S0: [K, V] initial state (values representable in the state dtype).
    tokens: list of dicts with keys q, k (K,), v (V,), a, b (scalars) and
        optionally z (V,).  All values must be bf16-exact.
    The read slot is state_indices[0, max(acc-1, 0)]; token t writes slot t+1.
    Returns dict(out [T, V], states [T, K, V], pool, idx).
    """
    S0 = np.asarray(S0, dtype=np.float64)
    K, V = S0.shape
    T = len(tokens)
    gated = "z" in tokens[0]
    q = bf16_bits(np.stack([t["q"] for t in tokens]).reshape(T, 1, K))
    k = bf16_bits(np.stack([t["k"] for t in tokens]).reshape(T, 1, K))
    v = bf16_bits(np.stack([t["v"] for t in tokens]).reshape(T, 1, V))
    a = bf16_bits(np.array([[t["a"]] for t in tokens]))
    b = bf16_bits(np.array([[t["b"]] for t in tokens]))
    z = bf16_bits(np.stack([t["z"] for t in tokens]).reshape(T, 1, V)) if gated else None
    w = bf16_bits(np.ones(V) if norm_w is None else norm_w) if gated else None
    idx = (np.arange(T, dtype=np.int32) + 1).reshape(1, T)
    read = max(acc - 1, 0)
    num_slots = T + 1
    if state_dtype == orc.F64:
        pool = np.zeros((num_slots, 1, K, V))
        pool[idx[0, read], 0] = S0
    elif state_dtype == orc.F32:
        pool = np.zeros((num_slots, 1, K, V), dtype=np.float32)
        pool[idx[0, read], 0] = S0.astype(np.float32)
    else:
        raise ValueError("use F64 or F32 here")
    res = orc.spec_decode(
        q=q, k=k, v=v, a=a, b=b, z=z, A_log=np.array([A_log], dtype=np.float32),
        dt_bias=bf16_bits(np.array([dt_bias])), norm_w=w, pool=pool,
        state_dtype=state_dtype, state_indices=idx,
        num_accepted=np.array([acc], dtype=np.int32),
        cu_seqlens=np.array([0, T], dtype=np.int32), scale=scale, eps=eps,
        states_T=T, num_threads=num_threads)
    return {"out": res["out_f64"][:, 0, :], "out_bf16": res["out_bf16"][:, 0, :],
            "states": res["states"][0, 0], "pool": pool, "idx": idx}


def initial_pool(case, slot_map=None):
    """Host pool for the oracle holding the case's touched slots.

    Without slot_map the pool has case.num_slots slots (untouched ones zero);
    with slot_map (compact pool) slot j holds the original slot slot_map[j].
    """
    if slot_map is None:
        touched = case.touched_slots()
        dt = np.float32 if case.state_dtype == orc.F32 else np.uint16
        pool = np.zeros((case.num_slots, case.H_v, case.K, case.V), dtype=dt)
        if len(touched):
            pool[touched] = case.slot_values(touched)
        return pool
    return np.ascontiguousarray(case.slot_values(slot_map))

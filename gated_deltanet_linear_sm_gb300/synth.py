"""Seeded synthetic inputs for the Gated DeltaNet speculative/MTP decode step.

This module only draws random numbers and lays them out; it contains none of
the arithmetic of the method.  Both the CUDA path (tests, ``bench.py``) and the
FP64 oracle consume what it produces, so the two sides always see the same
bits.

Value distributions (every config): q, k, v, z, a, b ~ N(0, 1) stored as
bf16; A_log = log U(1, 16) stored as fp32; dt_bias ~ N(0, 1) as bf16;
norm_w ~ N(1, 0.1) as bf16; state-pool slots ~ N(0, 0.1) in the state dtype.
Draw order for the token and parameter tensors: q, k, v, z, a, b, A_log,
dt_bias, norm_w, then lengths / acceptance / slots / gather rows.

State-pool slots are drawn per slot from an independent stream seeded by
``(seed, 1, slot)``, so the contents of any subset of a multi-GiB pool can be
produced without materialising the whole pool on the host.

Layouts (row-major, contiguous):
  q, k      [num_tokens, H_k, K]     bf16 bits (uint16)
  v, z, out [num_tokens, H_v, V]     bf16 bits (uint16)
  a, b      [num_tokens, H_v]        bf16 bits
  A_log     [H_v]                    float32
  dt_bias   [H_v]                    bf16 bits
  norm_w    [V]                      bf16 bits
  pool      [num_slots, H_v, K, V]   state dtype (V contiguous)
  state_indices [batch, spec_stride] int32 (-1 = padded slot)
  num_accepted  [batch]              int32
  cu_seqlens    [batch + 1]          int32
  spec_token_indx [cu_seqlens[-1]]   int32 or None
"""
from __future__ import annotations

import dataclasses

import numpy as np

# state dtype codes (same numbering as gdn_dtype in include/gdnspec.h)
F32, BF16, F16 = 0, 1, 2
STATE_BYTES = {F32: 4, BF16: 2, F16: 2}
STATE_NAMES = {F32: "f32", BF16: "bf16", F16: "f16"}


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (library conversion) and return the bits."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def f32_to_f16_bits(x: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def _to_state_bits(x: np.ndarray, state_dtype: int) -> np.ndarray:
    if state_dtype == F32:
        return np.ascontiguousarray(x, dtype=np.float32)
    if state_dtype == BF16:
        return f32_to_bf16_bits(x)
    if state_dtype == F16:
        return f32_to_f16_bits(x)
    raise ValueError(f"unknown state dtype {state_dtype}")


@dataclasses.dataclass
class Case:
    """One synthetic batch for one speculative decode step of one layer."""

    name: str
    batch: int
    num_tokens: int
    H_k: int
    H_v: int
    K: int
    V: int
    spec_stride: int
    max_T: int
    num_slots: int
    state_dtype: int
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    a: np.ndarray
    b: np.ndarray
    z: np.ndarray | None
    A_log: np.ndarray
    dt_bias: np.ndarray
    norm_w: np.ndarray | None
    state_indices: np.ndarray
    num_accepted: np.ndarray
    cu_seqlens: np.ndarray
    spec_token_indx: np.ndarray | None
    seed: int = 0
    scale: float = 128 ** -0.5
    eps: float = 1e-5
    pool_std: float = 0.1

    # ---- pool contents -------------------------------------------------
    @property
    def slot_elems(self) -> int:
        return self.H_v * self.K * self.V

    @property
    def slot_bytes(self) -> int:
        return self.slot_elems * STATE_BYTES[self.state_dtype]

    def slot_values(self, slots) -> np.ndarray:
        """Initial contents of the given slots, in the state dtype's bits.

        Shape [len(slots), H_v, K, V]; float32 for fp32 state, uint16 bits
        for bf16 / fp16 state.
        """
        slots = [int(s) for s in slots]
        out = np.empty((len(slots), self.slot_elems), dtype=np.float32)
        for n, s in enumerate(slots):
            rng = np.random.default_rng([self.seed, 1, s])
            out[n] = rng.normal(0.0, self.pool_std, self.slot_elems).astype(np.float32)
        bits = _to_state_bits(out, self.state_dtype)
        return bits.reshape(len(slots), self.H_v, self.K, self.V)

    # ---- index bookkeeping (plain integer work) ---------------------------
    def q_lens(self) -> np.ndarray:
        return np.diff(self.cu_seqlens.astype(np.int64))

    def read_slots(self) -> np.ndarray:
        """Slot each sequence starts from (-1 for padded / empty sequences)."""
        out = np.full(self.batch, -1, dtype=np.int64)
        ql = self.q_lens()
        for i in range(self.batch):
            if ql[i] <= 0:
                continue
            j = max(int(self.num_accepted[i]) - 1, 0)
            out[i] = int(self.state_indices[i, j])
        return out

    def touched_slots(self) -> np.ndarray:
        """Sorted unique non-negative slots that the step reads or writes."""
        ql = self.q_lens()
        rs = self.read_slots()
        s = set()
        for i in range(self.batch):
            if ql[i] <= 0 or rs[i] < 0:
                continue
            s.add(int(rs[i]))
            for t in range(int(ql[i])):
                w = int(self.state_indices[i, t])
                if w >= 0:
                    s.add(w)
        return np.array(sorted(s), dtype=np.int64)

    def token_rows(self) -> np.ndarray:
        """Row of the token tensors that each spec token occupies."""
        n = int(self.cu_seqlens[-1])
        if self.spec_token_indx is None:
            return np.arange(n, dtype=np.int64)
        return self.spec_token_indx.astype(np.int64)


def _bf16(rng: np.random.Generator, shape, loc=0.0, scale=1.0) -> np.ndarray:
    return f32_to_bf16_bits(rng.normal(loc, scale, shape).astype(np.float32))


def make_case(
    *,
    name: str = "custom",
    batch: int,
    H_k: int,
    H_v: int,
    T: int,
    state_dtype: int,
    num_slots: int,
    K: int = 128,
    V: int = 128,
    spec_stride: int | None = None,
    q_lens=None,
    acc="uniform",
    pad_prob: float = 0.0,
    extra_rows: int = 0,
    gated: bool = True,
    A_log_range=(1.0, 16.0),
    seed: int = 0,
) -> Case:
    """General seeded case.

    q_lens: None (every sequence has T draft tokens), "ragged" (U{0..T}),
        or an explicit list.
    acc: "uniform" (U{0..T}), "binomial" (Binomial(T, 0.7) clamped to [0, T]),
        or an explicit list.
    pad_prob: probability that each slot entry is -1 (CUDA-graph padding).
    extra_rows: non-spec token rows interleaved with the spec rows; when > 0
        the spec rows are gathered through spec_token_indx.
    A_log_range: A_log = log U(lo, hi); the default gives per-token decays
        of about e^-0.7 .. e^-11, a small range such as (1e-3, 5e-2) keeps the
        state alive over hundreds of tokens (long-prompt cases).
    """
    rng = np.random.default_rng(seed)
    stride = T if spec_stride is None else spec_stride
    if q_lens is None:
        ql = np.full(batch, T, dtype=np.int64)
    elif isinstance(q_lens, str) and q_lens == "ragged":
        ql = None  # drawn below, after the tensors, to keep the draw order
    else:
        ql = np.asarray(q_lens, dtype=np.int64)
    # token counts are needed before drawing the token tensors
    if ql is None:
        ql_rng = np.random.default_rng([seed, 2])
        ql = ql_rng.integers(0, T + 1, size=batch).astype(np.int64)
    n_spec = int(ql.sum())
    num_tokens = n_spec + int(extra_rows)

    q = _bf16(rng, (num_tokens, H_k, K))
    k = _bf16(rng, (num_tokens, H_k, K))
    v = _bf16(rng, (num_tokens, H_v, V))
    z = _bf16(rng, (num_tokens, H_v, V))
    a = _bf16(rng, (num_tokens, H_v))
    b = _bf16(rng, (num_tokens, H_v))
    A_log = np.log(rng.uniform(A_log_range[0], A_log_range[1], H_v)).astype(np.float32)
    dt_bias = _bf16(rng, (H_v,))
    norm_w = _bf16(rng, (V,), 1.0, 0.1)

    if isinstance(acc, str) and acc == "uniform":
        num_acc = rng.integers(0, T + 1, size=batch)
    elif isinstance(acc, str) and acc == "binomial":
        num_acc = np.clip(rng.binomial(T, 0.7, size=batch), 0, T)
    else:
        num_acc = np.asarray(acc)
    num_acc = num_acc.astype(np.int32)

    if batch * stride > num_slots:
        raise ValueError("pool too small for distinct slots")
    perm = rng.permutation(num_slots)
    idx = perm[: batch * stride].reshape(batch, stride).astype(np.int32)
    if pad_prob > 0:
        pad = rng.random((batch, stride)) < pad_prob
        idx[pad] = -1
    cu = np.zeros(batch + 1, dtype=np.int32)
    cu[1:] = np.cumsum(ql)
    if extra_rows > 0:
        rows = np.sort(rng.choice(num_tokens, size=n_spec, replace=False)).astype(np.int32)
    else:
        rows = None
    return Case(
        name=name, batch=batch, num_tokens=num_tokens, H_k=H_k, H_v=H_v, K=K, V=V,
        spec_stride=stride, max_T=max(int(ql.max()) if batch else 1, 1),
        num_slots=num_slots, state_dtype=state_dtype,
        q=q, k=k, v=v, a=a, b=b, z=z if gated else None, A_log=A_log,
        dt_bias=dt_bias, norm_w=norm_w if gated else None,
        state_indices=idx, num_accepted=num_acc, cu_seqlens=cu,
        spec_token_indx=rows, seed=seed,
    )


# ---- the five named workloads -------------------------------------------


def tiny(seed: int = 0) -> Case:
    """2 sequences, H_k=1, H_v=8, T=2, acceptance [1, 2], fp32 pool of 8 slots."""
    c = make_case(name="tiny", batch=2, H_k=1, H_v=8, T=2, state_dtype=F32,
                  num_slots=8, acc=[1, 2], seed=seed)
    return c


def decode_batch(seed: int = 0) -> Case:
    """BS=32, H_k=2, H_v=16, T=4, bf16 state, acceptance U{0..4}, 4*BS*T slots."""
    return make_case(name="decode_bs32_t4_bf16", batch=32, H_k=2, H_v=16, T=4,
                     state_dtype=BF16, num_slots=4 * 32 * 4, seed=seed)


def sweep_num_slots(bs: int, T: int, state_dtype: int, H_v: int = 16) -> int:
    """max(4*BS*T, ceil(2 GiB / slot_bytes)): the pool is at least 2 GiB."""
    slot_bytes = H_v * 128 * 128 * STATE_BYTES[state_dtype]
    return max(4 * bs * T, -(-(2 << 30) // slot_bytes))


def sweep(bs: int, state_dtype: int, T: int = 8, seed: int = 0,
          num_slots: int | None = None) -> Case:
    """Batch sweep point: H_k=2, H_v=16, T=8, ragged acceptance, >=2 GiB pool."""
    ns = sweep_num_slots(bs, T, state_dtype) if num_slots is None else num_slots
    return make_case(name=f"sweep_bs{bs}_t{T}_{STATE_NAMES[state_dtype]}", batch=bs,
                     H_k=2, H_v=16, T=T, state_dtype=state_dtype, num_slots=ns,
                     seed=seed)


def mixed(seed: int = 0) -> Case:
    """48 spec sequences (T=3) among 80 non-spec rows, 10% padded slots, fp16 state."""
    return make_case(name="mixed_48x3_plus80_f16", batch=48, H_k=2, H_v=16, T=3,
                     state_dtype=F16, num_slots=576, pad_prob=0.1, extra_rows=80,
                     seed=seed)


def large(seed: int = 0, num_slots: int = 8192) -> Case:
    """BS=256, H_k=4, H_v=32, T=8, bf16 state, 8192-slot pool, Binomial(8, 0.7)."""
    return make_case(name="large_bs256_t8_bf16", batch=256, H_k=4, H_v=32, T=8,
                     state_dtype=BF16, num_slots=num_slots, acc="binomial", seed=seed)


def disjoint_index_sets(case: Case, n_sets: int, seed: int = 1) -> list[np.ndarray]:
    """n_sets slot tables with the same shape as case.state_indices, pairwise
    disjoint, each with the same -1 pattern as the case's own table.  Rotating
    through them between timed steps keeps the touched state out of L2."""
    rng = np.random.default_rng([case.seed, seed, 3])
    B, S = case.state_indices.shape
    need = n_sets * B * S
    if need > case.num_slots:
        raise ValueError(f"{n_sets} disjoint sets need {need} slots > {case.num_slots}")
    perm = rng.permutation(case.num_slots)[:need].astype(np.int32).reshape(n_sets, B, S)
    pad = case.state_indices < 0
    out = []
    for n in range(n_sets):
        t = perm[n].copy()
        t[pad] = -1
        out.append(t)
    return out


def subset(case: Case, seqs) -> tuple[Case, np.ndarray, np.ndarray]:
    """A case holding only the given sequences, with a compact pool.

    Returns (sub_case, slot_map, rows): slot_map[j] is the original slot of the
    sub-case's slot j, rows[n] the original token row of the sub-case's row n.  Sequences are independent, so the sub-case's results
    equal the corresponding part of the full case's results.  Token rows keep
    their original numbering only through spec_token_indx: the sub-case holds
    the selected rows contiguously.
    """
    seqs = [int(s) for s in seqs]
    cu = case.cu_seqlens.astype(np.int64)
    rows_all = case.token_rows()
    rows = []
    new_cu = [0]
    for i in seqs:
        rows.extend(rows_all[cu[i]:cu[i + 1]].tolist())
        new_cu.append(len(rows))
    rows = np.array(rows, dtype=np.int64)
    idx = case.state_indices[seqs].astype(np.int64)
    used = sorted({int(s) for s in idx.ravel() if s >= 0})
    remap = {s: j for j, s in enumerate(used)}
    new_idx = np.array([[remap[int(s)] if s >= 0 else -1 for s in row] for row in idx],
                       dtype=np.int32).reshape(idx.shape)
    sub = dataclasses.replace(
        case,
        name=case.name + "_subset",
        batch=len(seqs),
        num_tokens=len(rows),
        q=case.q[rows], k=case.k[rows], v=case.v[rows], a=case.a[rows], b=case.b[rows],
        z=None if case.z is None else case.z[rows],
        state_indices=new_idx,
        num_accepted=case.num_accepted[seqs].copy(),
        cu_seqlens=np.array(new_cu, dtype=np.int32),
        spec_token_indx=None,
        num_slots=max(len(used), 1),
    )
    return sub, np.array(used, dtype=np.int64), rows


def algorithmic_bytes(case: Case, out_bytes: int = 2) -> int:
    """Bytes the step must move: one state-tile read per active (sequence,
    v-head), one tile write per valid slot write, and the token rows
    (q, k per k-head; v, z, out per v-head; a, b per v-head), plus parameters
    and the index tensors."""
    s = STATE_BYTES[case.state_dtype]
    tile = case.K * case.V * s
    ql = case.q_lens()
    rs = case.read_slots()
    state = 0
    tokens = 0
    for i in range(case.batch):
        if ql[i] <= 0 or rs[i] < 0 or rs[i] >= case.num_slots:
            continue
        n_w = sum(1 for t in range(int(ql[i])) if 0 <= case.state_indices[i, t] < case.num_slots)
        state += case.H_v * tile * (1 + n_w)
        tokens += int(ql[i])
    # v and out always; z only in gated mode
    per_token = case.H_k * 2 * case.K * 2 + case.H_v * (case.V * 2 * (2 + (1 if case.z is not None else 0)) + 2 * 2)
    params = case.H_v * (4 + 2) + (case.V * 2 if case.norm_w is not None else 0)
    index = 4 * (2 * case.batch + 1 + case.batch * case.spec_stride
                 + (int(case.cu_seqlens[-1]) if case.spec_token_indx is not None else 0))
    return state + tokens * per_token + params + index


def token_head_updates(case: Case) -> int:
    """Draft-token x v-head updates one step performs (active sequences only)."""
    ql = case.q_lens()
    rs = case.read_slots()
    n = 0
    for i in range(case.batch):
        if ql[i] > 0 and 0 <= rs[i] < case.num_slots:
            n += int(ql[i])
    return n * case.H_v


# ---- inputs of the short causal convolution in front of the step ----------


@dataclasses.dataclass
class ConvInputs:
    """Pre-convolution projection rows and conv state for a Case.

    x          [num_tokens, conv_dim]              bf16 bits, channels q | k | v
    weight     [conv_dim, width]                   bf16 bits
    bias       [conv_dim]                          bf16 bits, or None
    pool       [num_conv_slots, state_len, conv_dim] bf16 bits
    conv_in, conv_out  [batch]                     int32, disjoint sets of slots
    """
    width: int
    state_len: int
    x: np.ndarray
    weight: np.ndarray
    bias: np.ndarray | None
    pool: np.ndarray
    conv_in: np.ndarray
    conv_out: np.ndarray

    @property
    def conv_dim(self) -> int:
        return int(self.x.shape[1])


def conv_inputs(case: Case, width: int = 4, num_conv_slots: int | None = None, with_bias: bool = True,
                seed: int = 0) -> ConvInputs:
    """x ~ N(0, 1), weight ~ N(0, 0.5), bias ~ N(0, 0.1), conv-state rows
    ~ N(0, 1), all bf16; state_len = width - 1 + spec_stride; read and write
    slots drawn without replacement (read slots first)."""
    rng = np.random.default_rng([seed, 3])
    D = 2 * case.H_k * case.K + case.H_v * case.V
    ns = num_conv_slots if num_conv_slots is not None else max(2 * case.batch, 2)
    if ns < 2 * case.batch:
        raise ValueError("need two conv slots per sequence")
    state_len = width - 1 + case.spec_stride
    x = _bf16(rng, (case.num_tokens, D))
    weight = _bf16(rng, (D, width), 0.0, 0.5)
    bias = _bf16(rng, (D,), 0.0, 0.1) if with_bias else None
    pool = _bf16(rng, (ns, state_len, D))
    perm = rng.permutation(ns).astype(np.int32)
    return ConvInputs(width=width, state_len=state_len, x=x, weight=weight, bias=bias, pool=pool,
                      conv_in=perm[:case.batch].copy(), conv_out=perm[case.batch:2 * case.batch].copy())


def conv_algorithmic_bytes(case: Case, ci: ConvInputs, out_bytes: int = 2) -> int:
    """algorithmic_bytes of the step (x rows hold the same channels as q, k, v)
    plus, per processed sequence, the W-1 history rows read, the W-1+q_len
    rows of the new conv slot written, and the conv weights, bias and slot
    indices once."""
    D, W = ci.conv_dim, ci.width
    ql = case.q_lens()
    rs = case.read_slots()
    conv = 0
    for i in range(case.batch):
        if ql[i] <= 0 or rs[i] < 0 or rs[i] >= case.num_slots:
            continue
        if ci.conv_in[i] >= 0:
            conv += (W - 1) * D * 2
        if ci.conv_out[i] >= 0:
            conv += (W - 1 + int(ql[i])) * D * 2
    conv += D * W * 2 + (D * 2 if ci.bias is not None else 0) + 8 * case.batch
    return algorithmic_bytes(case, out_bytes) + conv

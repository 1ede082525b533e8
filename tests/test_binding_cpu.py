"""The Python binding's marshalling without a GPU: sizes and row strides in
gdn_dims, the packed mixed_qkv views, and the refusals that happen before the
library is called."""
from __future__ import annotations

import pytest
import torch

from gated_deltanet_linear_sm_gb300 import binding

H_K, H_V, K = 2, 16, 128


def _tensors(N=5, B=2, S=3, slots=8):
    bf = torch.bfloat16
    return dict(
        q=torch.zeros(N, H_K, K, dtype=bf), k=torch.zeros(N, H_K, K, dtype=bf),
        v=torch.zeros(N, H_V, K, dtype=bf), a=torch.zeros(N, H_V, dtype=bf), b=torch.zeros(N, H_V, dtype=bf),
        z=torch.zeros(N, H_V, K, dtype=bf), out=torch.zeros(N, H_V, K, dtype=bf),
        pool=torch.zeros(slots, H_V, K, K, dtype=bf), idx=torch.zeros(B, S, dtype=torch.int32))


def test_dense_dims():
    t = _tensors()
    d = binding.make_dims(t["q"], t["v"], t["pool"], t["idx"], k=t["k"], a=t["a"], b=t["b"], z=t["z"],
                          out=t["out"], max_T=2, split=0)
    assert (d.batch, d.num_tokens, d.H_k, d.H_v, d.K, d.V) == (2, 5, H_K, H_V, K, K)
    assert (d.spec_stride, d.max_T, d.num_slots, d.split, d.flags) == (3, 2, 8, 0, 0)
    assert (d.q_stride, d.k_stride, d.v_stride) == (H_K * K, H_K * K, H_V * K)
    assert (d.a_stride, d.b_stride, d.z_stride, d.out_stride) == (H_V, H_V, H_V * K, H_V * K)


def test_max_T_defaults_to_the_slot_columns():
    t = _tensors(S=5)
    assert binding.make_dims(t["q"], t["v"], t["pool"], t["idx"]).max_T == 5
    # a slot table wider than the 8-token limit: the default stays at 8
    t = _tensors(S=12)
    assert binding.make_dims(t["q"], t["v"], t["pool"], t["idx"]).max_T == 8


def test_packed_mixed_qkv_views_carry_the_packed_row_stride():
    """q, k, v as views into one [N, 2 H_k K + H_v V] tensor (channels q | k | v)."""
    N = 4
    row = 2 * H_K * K + H_V * K
    packed = torch.zeros(N, row, dtype=torch.bfloat16)
    q = packed[:, :H_K * K].view(N, H_K, K)
    k = packed[:, H_K * K:2 * H_K * K].view(N, H_K, K)
    v = packed[:, 2 * H_K * K:].view(N, H_V, K)
    t = _tensors(N=N)
    d = binding.make_dims(q, v, t["pool"], t["idx"], k=k)
    assert (d.q_stride, d.k_stride, d.v_stride) == (row, row, row)


def test_one_token_uses_the_dense_stride():
    """With one row the stride between rows is meaningless; the dense one is passed."""
    t = _tensors(N=1)
    q = torch.zeros(1, H_K * K + 64, dtype=torch.bfloat16)[:, :H_K * K].view(1, H_K, K)   # padded row
    assert binding.make_dims(q, t["v"], t["pool"], t["idx"]).q_stride == H_K * K


def test_non_contiguous_heads_are_refused():
    t = _tensors()
    q = torch.zeros(5, K, H_K, dtype=torch.bfloat16).transpose(1, 2)   # head dim strided
    with pytest.raises(ValueError):
        binding.make_dims(q, t["v"], t["pool"], t["idx"])
    a = torch.zeros(H_V, 5, dtype=torch.bfloat16).t()
    with pytest.raises(ValueError):
        binding.make_dims(t["q"], t["v"], t["pool"], t["idx"], a=a)


def test_prepare_refuses_host_tensors_before_any_library_call():
    t = _tensors()
    f32 = torch.zeros(H_V, dtype=torch.float32)
    i32 = torch.zeros(3, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA"):
        binding.prepare(t["q"], t["k"], t["v"], t["a"], t["b"], t["z"], f32, t["a"][0], torch.zeros(K),
                        t["pool"], t["idx"], i32[:2], i32, t["out"])


def _params():
    return dict(A_log=torch.zeros(H_V, dtype=torch.float32), dt_bias=torch.zeros(H_V, dtype=torch.bfloat16),
                norm_w=torch.zeros(K, dtype=torch.bfloat16))


BAD_SHAPES = {
    "a": lambda t, p: t.update(a=torch.zeros(5, H_V // 2, dtype=torch.bfloat16)),
    "b": lambda t, p: t.update(b=torch.zeros(4, H_V, dtype=torch.bfloat16)),
    "z": lambda t, p: t.update(z=torch.zeros(5, H_V // 2, K, dtype=torch.bfloat16)),
    "out": lambda t, p: t.update(out=torch.zeros(4, H_V, K, dtype=torch.bfloat16)),
    "dt_bias": lambda t, p: p.update(dt_bias=torch.zeros(H_V - 1, dtype=torch.bfloat16)),
    "A_log": lambda t, p: p.update(A_log=torch.zeros(H_V // 2, dtype=torch.float32)),
    "norm_w": lambda t, p: p.update(norm_w=torch.zeros(K // 2, dtype=torch.bfloat16)),
    "v": lambda t, p: t.update(v=torch.zeros(6, H_V, K, dtype=torch.bfloat16)),
}


@pytest.mark.parametrize("field", sorted(BAD_SHAPES))
def test_mismatched_sizes_are_refused_before_the_library(field, monkeypatch):
    """A short a / b / z / out / dt_bias / A_log / norm_w (or a v with the wrong
    token count) is refused by every entry point before the library is loaded
    or called: the kernels would read or write past the end of such buffers."""
    def no_library():
        raise AssertionError("the library was reached")
    monkeypatch.setattr(binding, "load_library", no_library)
    t, p = _tensors(), _params()
    BAD_SHAPES[field](t, p)
    i32 = torch.zeros(3, dtype=torch.int32)
    with pytest.raises(ValueError, match="expected"):
        binding.prepare(t["q"], t["k"], t["v"], t["a"], t["b"], t["z"], p["A_log"], p["dt_bias"], p["norm_w"],
                        t["pool"], t["idx"], i32[:2], i32, t["out"])
    with pytest.raises(ValueError, match="expected"):
        binding.gdn_prefill(t["q"], t["k"], t["v"], t["a"], t["b"], t["z"], p["A_log"], p["dt_bias"],
                            p["norm_w"], t["pool"], i32[:2], i32[:2], i32, t["out"])
    with pytest.raises(ValueError, match="expected"):
        binding.gdn_prefill_chunked(t["q"], t["k"], t["v"], t["a"], t["b"], t["z"], p["A_log"], p["dt_bias"],
                                    p["norm_w"], t["pool"], i32[:2], i32[:2], i32, t["out"])
    if field != "v":
        D = 2 * H_K * K + H_V * K
        x = torch.zeros(5, D, dtype=torch.bfloat16)
        w = torch.zeros(D, 4, dtype=torch.bfloat16)
        cpool = torch.zeros(4, 6, D, dtype=torch.bfloat16)
        with pytest.raises(ValueError, match="expected"):
            binding.gdn_spec_decode_conv(x, w, None, cpool, i32[:2], i32[:2], t["a"], t["b"], t["z"],
                                         p["A_log"], p["dt_bias"], p["norm_w"], t["pool"], t["idx"], i32[:2],
                                         i32, t["out"], H_k=H_K)

"""The C-ABI boundary without a GPU: the library loads, exports every symbol
include/gdnspec.h declares, its ctypes mirror matches the C struct layout,
and host-side validation rejects bad arguments before anything is launched
(these calls return before any CUDA API is touched)."""
from __future__ import annotations

import ctypes
import os
import re
import subprocess

import pytest

import gated_deltanet_linear_sm_gb300 as gdn
from gated_deltanet_linear_sm_gb300 import binding
from gated_deltanet_linear_sm_gb300 import build as gbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdnspec.h")


@pytest.fixture(scope="module")
def lib():
    gbuild.build()
    return gdn.load_library()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"GDNSPEC_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)


def test_header_declares_the_entry_points():
    names = declared_functions()
    assert {"gdn_spec_decode", "gdn_spec_decode_split", "gdn_status_str", "gdn_version"} <= set(names)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(declared_functions()) == set(binding.EXPORTS)


def test_exports_are_only_the_c_abi(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", gdn.library_path()], capture_output=True, text=True)
    if out.returncode != 0:
        pytest.skip("nm not available")
    ours = [l.split()[-1] for l in out.stdout.splitlines() if l.split() and l.split()[-1].startswith("gdn_")]
    assert set(ours) == set(declared_functions())


def test_version_and_status_strings(lib):
    text = open(HEADER).read()
    want = int(re.search(r"#define GDNSPEC_VERSION (\d+)", text).group(1))
    assert gdn.version() == want
    for code in range(6):
        assert isinstance(gdn.status_str(code), str) and gdn.status_str(code)
    assert gdn.status_str(99) == "unknown status"


@pytest.mark.parametrize("struct", ["gdn_dims", "gdn_conv_dims"])
def test_dims_struct_layout_matches_c(tmp_path, struct):
    """Compile a probe against the header and compare sizeof / offsetof with
    the ctypes mirror."""
    mirror = getattr(binding, struct)
    fields = [f for f, _ in mirror._fields_]
    src = tmp_path / "probe.c"
    src.write_text(
        '#include <stdio.h>\n#include <stddef.h>\n#include "gdnspec.h"\nint main(void){\n'
        f'  printf("%zu\\n", sizeof({struct}));\n'
        + "".join(f'  printf("%zu\\n", offsetof({struct}, {f}));\n' for f in fields)
        + "  return 0;\n}\n")
    exe = tmp_path / "probe"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    vals = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    assert vals[0] == ctypes.sizeof(mirror)
    for f, off in zip(fields, vals[1:]):
        assert getattr(mirror, f).offset == off, f


def _dims(**over):
    d = binding.gdn_dims()
    d.batch, d.num_tokens, d.H_k, d.H_v, d.K, d.V = 2, 4, 1, 8, 128, 128
    d.spec_stride, d.max_T, d.num_slots = 2, 2, 8
    for k, v in over.items():
        setattr(d, k, v)
    return d


def _call(lib, dims, *, ptr=0x1000, z=0x1000, w=0x1000, state_dtype=0):
    P = ptr
    return lib.gdn_spec_decode(P, P, P, P, P, z, P, P, w, P, P, P, P, None, P,
                               ctypes.byref(dims), 0.088, 1e-5, state_dtype, None, None)


@pytest.mark.parametrize("over,code", [
    (dict(K=64), 3), (dict(V=256), 3), (dict(H_v=12, H_k=8), 2), (dict(max_T=9), 2),
    (dict(max_T=0), 2), (dict(spec_stride=0), 2), (dict(batch=-1), 2), (dict(num_slots=0), 2),
    (dict(split=3), 3), (dict(split=0x101), 3), (dict(split=0x108), 3), (dict(split=0x100), 3),
    (dict(split=0x200), 3), (dict(split=0x204), 3), (dict(split=0x302), 3),
    (dict(flags=8), 2), (dict(flags=-1), 2), (dict(q_stride=-4), 2),
])
def test_bad_dims_rejected(lib, over, code):
    assert _call(lib, _dims(**over)) == code


def test_bad_pointers_and_dtype_rejected(lib):
    assert _call(lib, _dims(), ptr=0) == 1                 # NULL tensors
    assert _call(lib, _dims(), z=None) == 1                # z without norm_w
    assert _call(lib, _dims(), ptr=0x1004) == 4            # pool not 16-byte aligned
    assert _call(lib, _dims(q_stride=1026)) == 4           # q rows not 8-byte aligned
    assert _call(lib, _dims(), state_dtype=7) == 3
    assert lib.gdn_spec_decode(*([None] * 15), None, 0.1, 1e-5, 0, None, None) == 1


def test_empty_batch_is_a_no_op(lib):
    # nothing is validated beyond the sizes and nothing is launched
    assert _call(lib, _dims(batch=0), ptr=0) == 0


def test_explicit_split_is_reported(lib):
    for s in (1, 2, 4, 8, binding.GDN_SPLIT_NARROW | 2, binding.GDN_SPLIT_NARROW | 4, binding.GDN_SPLIT_HALFK | 1,
              binding.GDN_SPLIT_HALFK | 2):
        assert binding.chosen_split(_dims(split=s)) == s
    assert binding.chosen_split(_dims(K=64)) == 0
    assert binding.chosen_split(_dims(), 7) == 0


def test_automatic_split():
    """FP32 state: the half-K layout over 2-CTA clusters with at most 64
    units, in one 16-warp CTA with at most 128; everything else one CTA of 8
    warps per unit."""
    H2, H1 = binding.GDN_SPLIT_HALFK | 2, binding.GDN_SPLIT_HALFK | 1
    assert binding.chosen_split(_dims(batch=4, H_v=16), binding.F32) == H2
    assert binding.chosen_split(_dims(batch=5, H_v=16), binding.F32) == H1
    assert binding.chosen_split(_dims(batch=8, H_v=16), binding.F32) == H1
    assert binding.chosen_split(_dims(batch=9, H_v=16), binding.F32) == 1
    assert binding.chosen_split(_dims(batch=4, H_v=16), binding.BF16) == 1
    assert binding.chosen_split(_dims(batch=4, H_v=16), binding.F16) == 1


def _cdims(**over):
    c = binding.gdn_conv_dims()
    c.width, c.state_len, c.num_conv_slots, c.x_stride = 4, 5, 4, 0
    for k, v in over.items():
        if k == "reserved":
            c.reserved[0] = v
        else:
            setattr(c, k, v)
    return c


def _call_conv(lib, dims, cdims, *, ptr=0x1000, bias=0x1000, state_dtype=0):
    P = ptr
    return lib.gdn_spec_decode_conv(P, P, bias, P, P, P, ctypes.byref(cdims), P, P, P, P, P, P, P, P, P, P, None, P,
                                    ctypes.byref(dims), 0.088, 1e-5, state_dtype, None, None)


@pytest.mark.parametrize("over,code", [
    (dict(width=0), 2), (dict(width=5), 2), (dict(state_len=4), 2), (dict(num_conv_slots=0), 2),
    (dict(x_stride=-4), 2), (dict(reserved=1), 2), (dict(x_stride=1026), 4),
])
def test_conv_bad_dims_rejected(lib, over, code):
    assert _call_conv(lib, _dims(), _cdims(**over)) == code


def test_conv_bad_pointers_rejected(lib):
    assert _call_conv(lib, _dims(), _cdims(), ptr=0) == 1        # NULL tensors
    assert _call_conv(lib, _dims(), _cdims(), bias=0x1002) == 4   # bias not 8-byte aligned
    assert _call_conv(lib, _dims(split=2), _cdims()) == 3         # the fused path has no split
    assert _call_conv(lib, _dims(split=binding.GDN_SPLIT_NARROW | 2), _cdims()) == 3
    assert _call_conv(lib, _dims(flags=8), _cdims()) == 2                 # an unknown flag bit
    assert _call_conv(lib, _dims(batch=0), _cdims(), ptr=0) == 0  # empty batch: nothing launched
    assert lib.gdn_spec_decode_conv(*([None] * 6), None, *([None] * 12), ctypes.byref(_dims()), 0.1, 1e-5, 0,
                                    None, None) == 1


def test_pool_beyond_32bit_rows_is_unsupported(lib):
    """The slot writes address the pool as one 2-D tensor with 32-bit row
    coordinates: num_slots * H_v * 128 must stay below 2^31 (checked before
    anything touches the GPU)."""
    assert _call(lib, _dims(num_slots=(1 << 31) // (8 * 128))) == 3
    assert _call_conv(lib, _dims(num_slots=(1 << 31) // (8 * 128)), _cdims()) == 3


def test_prefill_entry_points_take_no_flags(lib):
    """The early-read flags are a decode-step feature; the prefill entry points
    reject any flag before launching anything."""
    P = 0x1000
    for name in ("gdn_prefill", "gdn_prefill_chunked"):
        fn = getattr(lib, name)
        assert fn(P, P, P, P, P, P, P, P, P, P, P, P, P, P, ctypes.byref(_dims(flags=1)), 0.088, 1e-5, 0,
                  None, None) == 2

"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function include/mh3_preattn.h declares, and rejects bad argument sets
before launching anything (flashinfer.diffusion_ops.minimax_h3_bf16_pre_attention,
Parameters: stride, alignment, shape and P rules)."""
import ctypes
import os
import re

import pytest

from norm_adaln_qkv_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mh3_preattn.h")

H = 5376


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(mh3_\w+)\s*\(", text, re.M)))


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(binding.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_library_has_no_oracle_dependency():
    # The product library is built from csrc/ only.
    for src in build.SOURCES:
        text = open(os.path.join(build.CSRC, src)).read()
        assert "oracle" not in text.lower()


def test_size_helpers(lib):
    assert binding.workspace_bytes(0) == 0
    assert binding.workspace_bytes(-5) == 0
    assert binding.workspace_bytes(3) == 3 * H * 2
    assert binding.out_bytes(7) == 7 * 21504 * 2


# A fake, 256-byte aligned "device" address: validate() never dereferences.
BASE = 1 << 40


def good_args(**over):
    a = dict(M=64, x=BASE, x_norm_weight=BASE + 0x1000, adaln_scale=BASE + 0x2000,
             scale_row_stride=6 * H, adaln_shift=BASE + 0x3000, shift_row_stride=6 * H, rows=9,
             adaln_index=BASE + 0x4000, qkv_weight=BASE + 0x5000, q_norm_weight=BASE + 0x6000,
             k_norm_weight=BASE + 0x7000, rope_cos_sin=BASE + 0x8000, S=64, rope_positions=None,
             P=2, eps=1e-5, qk_eps=None, workspace=None, out=BASE + 0x9000)
    a.update(over)
    return a


def validate(**over):
    return binding.mh3_preattn_validate(**good_args(**over))


def test_validate_accepts_good_arguments(lib):
    assert validate() == 0
    assert validate(rope_positions=BASE + 0xA000, S=1) == 0  # explicit positions: any S >= 1
    assert validate(workspace=BASE + 0xB000) == 0
    assert validate(M=0, x=None, adaln_index=None, out=None) == 0  # empty call
    for P in (1, 2, 4, 8):
        assert validate(P=P) == 0
    assert validate(scale_row_stride=H, shift_row_stride=H + 8) == 0
    assert validate(qk_eps=float("nan")) == 0 and validate(qk_eps=-1.0) == 0


@pytest.mark.parametrize("over,code", [
    (dict(M=-1), 1),
    (dict(M=(1 << 30) + 1), 1),
    (dict(P=3), 1), (dict(P=16), 1), (dict(P=0), 1),
    (dict(rows=0), 1),
    (dict(S=0, rope_positions=BASE + 0xA000), 1),
    (dict(S=63), 1),  # identity positions need S >= M
    (dict(eps=0.0), 1), (dict(eps=float("inf")), 1), (dict(eps=-1e-5), 1),
    (dict(qk_eps=0.0), 1), (dict(qk_eps=float("inf")), 1),
    (dict(scale_row_stride=H - 8), 1),
    (dict(shift_row_stride=H + 4), 2),
    (dict(x=None), 1), (dict(qkv_weight=None), 1), (dict(out=None), 1),
    (dict(adaln_index=None), 1), (dict(rope_cos_sin=None), 1),
    (dict(x=BASE + 8), 2), (dict(adaln_scale=BASE + 0x2002), 2), (dict(out=BASE + 0x9004), 2),
    (dict(workspace=BASE + 0xB008), 2), (dict(adaln_index=BASE + 0x4004), 2),
    (dict(rope_positions=BASE + 0xA004), 2), (dict(rope_cos_sin=BASE + 0x8008), 2),
])
def test_validate_rejects(lib, over, code):
    assert validate(**over) == code
    assert binding.last_error() != ""


def test_run_without_handle_is_rejected(lib):
    a = good_args()
    rc = lib.mh3_preattn_run(
        None, None, a["M"], a["x"], a["x_norm_weight"], a["adaln_scale"], a["scale_row_stride"],
        a["adaln_shift"], a["shift_row_stride"], a["rows"], a["adaln_index"], a["qkv_weight"],
        a["q_norm_weight"], a["k_norm_weight"], a["rope_cos_sin"], a["S"], None, a["P"], 1e-5,
        -1.0, None, a["out"])
    assert rc == 1
    assert "handle" in binding.last_error()


def op_args(**over):
    a = dict(M=64, attn_out=BASE, o_weight=BASE + 0x1000, gate=BASE + 0x2000,
             gate_row_stride=6 * H, gate_rows=9, gate_index=BASE + 0x3000,
             residual=BASE + 0x10000000, out=BASE + 0x20000000)
    a.update(over)
    return a


def op_validate(**over):
    return binding.mh3_out_proj_validate(**op_args(**over))


def test_out_proj_validate_accepts_good_arguments(lib):
    assert op_validate() == 0
    assert op_validate(out=BASE + 0x10000000) == 0  # out may be the residual itself
    assert op_validate(M=0, attn_out=None, gate_index=None, residual=None, out=None) == 0
    assert op_validate(gate_row_stride=H, gate_rows=1) == 0


@pytest.mark.parametrize("over,code", [
    (dict(M=-1), 1), (dict(gate_rows=0), 1), (dict(gate_row_stride=H - 8), 1),
    (dict(gate_row_stride=H + 4), 2), (dict(attn_out=None), 1), (dict(o_weight=None), 1),
    (dict(gate=None), 1), (dict(gate_index=None), 1), (dict(residual=None), 1),
    (dict(out=None), 1), (dict(attn_out=BASE + 8), 2), (dict(gate=BASE + 0x2002), 2),
    (dict(gate_index=BASE + 0x3002), 2), (dict(out=BASE + 0x20000008), 2),
    # partial overlap of out and residual (64 rows x 10752 B)
    (dict(out=BASE + 0x10000000 + 10752 * 3), 1),
])
def test_out_proj_validate_rejects(lib, over, code):
    assert op_validate(**over) == code
    assert binding.last_error() != ""


def mlp_args(**over):
    a = dict(M=64, x=BASE, x_norm_weight=BASE + 0x1000, adaln_scale=BASE + 0x2000,
             scale_row_stride=6 * H, adaln_shift=BASE + 0x3000, shift_row_stride=6 * H,
             gate=BASE + 0x4000, gate_row_stride=6 * H, rows=9, adaln_index=BASE + 0x5000,
             residual=BASE + 0x10000000, fc1_weight=BASE + 0x6000, fc2_weight=BASE + 0x7000,
             eps=1e-5, workspace_a=None, workspace_y=None, out=BASE + 0x20000000)
    a.update(over)
    return a


def test_mlp_validate(lib):
    v = lambda **o: binding.mh3_mlp_validate(**mlp_args(**o))  # noqa: E731
    assert v() == 0
    assert v(out=BASE + 0x10000000) == 0  # out is the residual
    assert v(out=BASE) == 0  # out is x
    assert v(M=0, x=None, adaln_index=None, residual=None, out=None) == 0
    assert v(workspace_a=BASE + 0x30000000, workspace_y=BASE + 0x40000000) == 0
    assert binding.load().mh3_mlp_workspace_y_bytes(3) == 3 * 14336 * 2
    for over, code in [(dict(rows=0), 1), (dict(gate_row_stride=H - 8), 1),
                       (dict(gate_row_stride=H + 4), 2), (dict(gate=None), 1),
                       (dict(fc1_weight=None), 1), (dict(fc2_weight=BASE + 0x7008), 2),
                       (dict(workspace_y=BASE + 0x40000004), 2), (dict(eps=0.0), 1),
                       (dict(out=BASE + 10752 * 2), 1), (dict(residual=None), 1)]:
        assert v(**over) == code, over


def test_binding_wrappers_marshal_without_a_gpu(monkeypatch):
    """Every wrapper of the binding hands its C call to the status check
    (_check(rc, name)); the Handle methods run against a stub library that
    records the call, so a marshalling slip fails here rather than on a GPU."""
    import ast
    tree = ast.parse(open(binding.__file__).read())
    for node in ast.walk(tree):
        if isinstance(node, ast.Call) and getattr(node.func, "id", "") == "_check":
            assert len(node.args) == 2, f"_check with {len(node.args)} arguments at line {node.lineno}"

    calls = []

    class Stub:
        def __getattr__(self, name):
            def f(*args):
                calls.append(name)
                return 0
            return f

    monkeypatch.setattr(binding, "load", lambda *a, **k: Stub())
    h = object.__new__(binding.Handle)
    h._h = binding._vp(1)
    h.set_test_stall(True)
    assert h.device_status(stream=0) == 0  # 0: the default stream, no torch stream needed
    assert calls == ["mh3_preattn_set_test_stall", "mh3_preattn_device_status"]

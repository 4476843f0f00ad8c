"""The C-ABI library loads, exports every function include/k3da.h declares,
and refuses out-of-contract calls on the host before touching the GPU (CPU
only: no compute call is made)."""
import ctypes
import os
import re

import pytest

import speculative_decoding_drafter_k3_gb300 as k3da
from speculative_decoding_drafter_k3_gb300 import build as kbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "k3da.h")


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return k3da.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(k3da_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    assert declared_functions() == sorted(k3da.EXPORTED)


def test_library_exports_every_declared_function(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert lib.k3da_version() >= 100


def test_error_strings(lib):
    for code in [0, -1, -2, -3, -4, 1, 2, 4]:
        assert lib.k3da_error_string(code)


FAKE = 0x10000  # aligned, never dereferenced: every case below fails a host check first


def call_attn(lib, **over):
    a = dict(out=FAKE, qkv=FAKE, pool=FAKE, num_pages=16, pt=FAKE, stride=4, lens=FAKE, R=8, B=8,
             Hq=6, Hkv=1, D=64, scale=0.125, ws=FAKE, ws_bytes=1 << 30, status=None)
    a.update(over)
    return lib.k3da_attn(a["out"], a["qkv"], a["pool"], a["num_pages"], a["pt"], a["stride"],
                         a["lens"], a["R"], a["B"], a["Hq"], a["Hkv"], a["D"], a["scale"], a["ws"],
                         a["ws_bytes"], a["status"], None)


@pytest.mark.parametrize("over,code", [
    (dict(out=None), k3da.EINVAL),
    (dict(qkv=None), k3da.EINVAL),
    (dict(pool=None), k3da.EINVAL),
    (dict(pt=None), k3da.EINVAL),
    (dict(lens=None), k3da.EINVAL),
    (dict(out=FAKE + 2), k3da.EINVAL),
    (dict(pool=FAKE + 8), k3da.EINVAL),
    (dict(pt=FAKE + 2), k3da.EINVAL),
    (dict(R=0), k3da.EINVAL),
    (dict(R=9), k3da.EINVAL),
    (dict(B=0), k3da.EINVAL),
    (dict(B=9), k3da.EINVAL),
    (dict(stride=0), k3da.EINVAL),
    (dict(stride=1 << 25), k3da.EINVAL),        # page_stride * 64 would overflow an int
    (dict(num_pages=0), k3da.EINVAL),
    (dict(num_pages=1 << 40), k3da.EINVAL),
    (dict(scale=0.0), k3da.EINVAL),
    (dict(scale=float("nan")), k3da.EINVAL),
    (dict(D=128), k3da.EUNSUPPORTED),
    (dict(Hq=8, Hkv=1), k3da.EUNSUPPORTED),
    (dict(Hq=12, Hkv=2), k3da.EUNSUPPORTED),
    (dict(Hq=24, Hkv=1), k3da.EUNSUPPORTED),
    (dict(ws=None), k3da.EWORKSPACE),
    (dict(ws=FAKE + 4), k3da.EWORKSPACE),
])
def test_host_checks_refuse_out_of_contract_calls(lib, over, code):
    assert call_attn(lib, **over) == code


def call_qknorm(lib, **over):
    a = dict(pos=FAKE, pos_dtype=k3da.POS_I32, qw=FAKE, kw=FAKE, eps=1e-5, base=10000.0)
    a.update(over)
    return lib.k3da_attn_qknorm(FAKE, FAKE, FAKE, 16, FAKE, 4, FAKE, 8, 8, 24, 4, 64, 0.125,
                                a["pos"], a["pos_dtype"], a["qw"], a["kw"], a["eps"], a["base"],
                                None, 1 << 30, None, None)


@pytest.mark.parametrize("over", [
    dict(pos=None), dict(qw=None), dict(kw=None), dict(pos_dtype=2),
    dict(pos=FAKE + 4, pos_dtype=k3da.POS_I64), dict(eps=-1.0), dict(eps=float("inf")),
    dict(base=1.0), dict(base=float("nan")),
])
def test_qknorm_host_checks(lib, over):
    assert call_qknorm(lib, **over) == k3da.EINVAL


def test_workspace_query_refuses_bad_sizes(lib):
    assert lib.k3da_workspace_bytes(0, 8, 6, 1, 32) == 0
    assert lib.k3da_workspace_bytes(8, 9, 6, 1, 32) == 0
    assert lib.k3da_workspace_bytes(8, 8, 6, 2, 32) == 0
    assert lib.k3da_workspace_bytes(8, 8, 6, 1, 0) == 0
    assert lib.k3da_workspace_bytes(8, 8, 6, 1, 1 << 25) == 0
    assert lib.k3da_workspace_bytes(8, 8, 6, 1, (1 << 25) - 1) > 0


def test_workspace_size_depends_on_shapes_only(lib):
    ws = lib.k3da_workspace_bytes
    assert ws(1, 8, 6, 1, 32) > 0
    # Block length never changes it; it grows with the page stride and the
    # number of (request, kv head) units once chunks reach their maximum.
    for R, Hq, Hkv in [(1, 6, 1), (8, 6, 1), (3, 24, 4), (8, 24, 4)]:
        assert ws(R, 8, Hq, Hkv, 32) == ws(R, 1, Hq, Hkv, 32) == ws(R, 5, Hq, Hkv, 32)
        assert ws(R, 8, Hq, Hkv, 2048) >= ws(R, 8, Hq, Hkv, 512) >= ws(R, 8, Hq, Hkv, 32)
    assert ws(8, 8, 24, 4, 2048) > ws(8, 8, 24, 4, 512) > ws(8, 8, 24, 4, 32)
    assert ws(8, 8, 24, 4, 2048) > ws(1, 8, 24, 4, 2048)
    # With long rows every unit has ceil((stride+1)/32) slots of the same size.
    slot = (ws(8, 8, 24, 4, 4096 - 1) - ws(8, 8, 24, 4, 2048 - 1)) // (32 * (128 - 64))
    assert slot == 48 * 64 * 2 + 48 * 8  # bf16 O and fp32 (m, l) per row
    assert ws(8, 8, 24, 4, 2048 - 1) - ws(4, 8, 24, 4, 2048 - 1) == 16 * 64 * slot


def test_product_path_does_not_touch_the_oracle():
    # The CUDA path and the oracle share no code: no import either way.
    pkg = os.path.join(ROOT, "speculative_decoding_drafter_k3_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".h", ".cuh", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, re.M), f
                assert "k3da_oracle" not in text and "k3o_" not in text, f
    for f in os.listdir(os.path.join(ROOT, "oracle")):
        if f.endswith((".py", ".c", ".h")):
            text = open(os.path.join(ROOT, "oracle", f)).read()
            assert "speculative_decoding_drafter_k3_gb300" not in text and "k3da.h" not in text, f


def call_norm_rope(lib, **over):
    a = dict(qkv=FAKE, T=64, Hq=6, Hkv=1, D=64, pos=FAKE, pos_dtype=k3da.POS_I64, qw=FAKE, kw=FAKE,
             eps=1e-5, base=10000.0)
    a.update(over)
    return lib.k3da_qk_norm_rope(a["qkv"], a["T"], a["Hq"], a["Hkv"], a["D"], a["pos"], a["pos_dtype"],
                                 a["qw"], a["kw"], a["eps"], a["base"], None)


@pytest.mark.parametrize("over,code", [
    (dict(qkv=None), k3da.EINVAL),
    (dict(pos=None), k3da.EINVAL),
    (dict(qw=None), k3da.EINVAL),
    (dict(kw=None), k3da.EINVAL),
    (dict(T=0), k3da.EINVAL),
    (dict(Hq=8, Hkv=1), k3da.EUNSUPPORTED),
    (dict(Hq=24, Hkv=1), k3da.EUNSUPPORTED),
    (dict(D=128), k3da.EUNSUPPORTED),
    (dict(pos_dtype=7), k3da.EINVAL),
    (dict(pos=FAKE + 4), k3da.EINVAL),          # int64 positions on a 4-byte boundary
    (dict(qkv=FAKE + 1), k3da.EINVAL),
    (dict(eps=float("nan")), k3da.EINVAL),
    (dict(eps=-1.0), k3da.EINVAL),
    (dict(base=1.0), k3da.EINVAL),
    (dict(base=float("inf")), k3da.EINVAL),
])
def test_norm_rope_refuses_out_of_contract_calls(lib, over, code):
    assert call_norm_rope(lib, **over) == code


def _yarn(**over):
    y = dict(factor=4.0, original_max_position=4096.0, beta_fast=32.0, beta_slow=1.0, mscale=1.1386)
    y.update(over)
    return k3da.Yarn(**y)


@pytest.mark.parametrize("over", [dict(factor=0.5), dict(factor=float("nan")), dict(original_max_position=0.0),
                                  dict(beta_fast=1.0), dict(beta_slow=0.0), dict(mscale=-1.0),
                                  dict(mscale=float("inf"))])
def test_yarn_calls_refuse_bad_scaling(lib, over):
    y = _yarn(**over)
    assert lib.k3da_qk_norm_rope_yarn(FAKE, 64, 6, 1, 64, FAKE, k3da.POS_I64, FAKE, FAKE, 1e-5, 10000.0,
                                      ctypes.byref(y), None) == k3da.EINVAL
    assert lib.k3da_attn_qknorm_yarn(FAKE, FAKE, FAKE, 16, FAKE, 4, FAKE, 8, 8, 6, 1, 64, 0.125, FAKE,
                                     k3da.POS_I64, FAKE, FAKE, 1e-5, 10000.0, ctypes.byref(y), FAKE, 1 << 30,
                                     None, None) == k3da.EINVAL


def test_yarn_calls_refuse_a_missing_spec(lib):
    assert lib.k3da_qk_norm_rope_yarn(FAKE, 64, 6, 1, 64, FAKE, k3da.POS_I64, FAKE, FAKE, 1e-5, 10000.0,
                                      None, None) == k3da.EINVAL
    assert lib.k3da_attn_qknorm_yarn(FAKE, FAKE, FAKE, 16, FAKE, 4, FAKE, 8, 8, 6, 1, 64, 0.125, FAKE,
                                     k3da.POS_I64, FAKE, FAKE, 1e-5, 10000.0, None, FAKE, 1 << 30,
                                     None, None) == k3da.EINVAL


def test_wait_selftest_refuses_bad_arguments(lib):
    assert lib.k3da_selftest_wait_timeout(None, 1000000, None) == k3da.EINVAL
    assert lib.k3da_selftest_wait_timeout(FAKE + 2, 1000000, None) == k3da.EINVAL
    assert lib.k3da_selftest_wait_timeout(FAKE, 0, None) == k3da.EINVAL
    assert lib.k3da_selftest_wait_timeout(FAKE, 3_000_000_000, None) == k3da.EINVAL


def test_binding_refuses_host_tensors_before_any_call(lib):
    import torch
    from speculative_decoding_drafter_k3_gb300 import workloads
    case = workloads.tiny()  # CPU tensors: the binding must refuse them, never fall back
    out = torch.empty(case.T, case.Hq * 64, dtype=torch.bfloat16)
    ws = torch.empty(1 << 20, dtype=torch.uint8)
    with pytest.raises(k3da.K3daError):
        k3da.k3da_attn(out, case.qkv, case.pool, case.page_table, case.ctx_lens, block_len=case.B,
                       num_q_heads=case.Hq, num_kv_heads=case.Hkv, workspace=ws)
    with pytest.raises(k3da.K3daError):
        k3da.k3da_qk_norm_rope(case.qkv, torch.zeros(case.T, dtype=torch.int64), torch.ones(64, dtype=torch.bfloat16),
                               torch.ones(64, dtype=torch.bfloat16), num_q_heads=6, num_kv_heads=1)


def test_workspace_query_through_the_binding(lib):
    n = k3da.workspace_bytes(8, 8, 24, 4, 2048)
    assert n == lib.k3da_workspace_bytes(8, 8, 24, 4, 2048) > 512
    with pytest.raises(k3da.K3daError):
        k3da.workspace_bytes(9, 8, 24, 4, 2048)

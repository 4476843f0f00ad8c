"""The entry point that allocates nothing (k3da_attn_qknorm_noalloc).

Some callers cannot allocate device memory: a host callback or a real-time
path where cudaMalloc is forbidden, or a plugin whose host framework owns
every device allocation and offers no workspace.  For them the library keeps
a fixed scratch array on each GPU.  These tests call that entry point through
the C ABI and require its output to equal, bit for bit, that of
k3da_attn_qknorm with a caller-owned workspace (the same kernels on the same
inputs, and reruns are bitwise), and to match the oracle element by element
(2e-2 absolute + 2e-2 relative).  Calls come in a row with other inputs and
other shapes in between, so stale scratch contents would show.  Sizes beyond
the array are refused.  Host-resident inputs work through it too.  Kept in
the last test file so a run that stops at the first failure has already run
every other test."""
import pytest
import torch

import speculative_decoding_drafter_k3_gb300 as k3da
from speculative_decoding_drafter_k3_gb300 import workloads
from common import assert_close, oracle_for

pytestmark = pytest.mark.gpu


def with_workspace(case):
    out = torch.empty(case.T, case.Hq * case.D, dtype=torch.bfloat16, device="cuda")
    ws = k3da.case_workspace(case)
    ws.fill_(0xFF)
    return k3da.k3da_attn_qknorm(out, case.qkv, case.pool, case.page_table, case.ctx_lens,
                                 case.positions, case.q_norm_w, case.k_norm_w, block_len=case.B,
                                 num_q_heads=case.Hq, num_kv_heads=case.Hkv, workspace=ws)


def without_allocation(case, status):
    out = torch.empty(case.T, case.Hq * case.D, dtype=torch.bfloat16, device="cuda")
    return k3da.k3da_attn_qknorm_noalloc(out, case.qkv, case.pool, case.page_table, case.ctx_lens,
                                         case.positions, case.q_norm_w, case.k_norm_w,
                                         block_len=case.B, num_q_heads=case.Hq,
                                         num_kv_heads=case.Hkv, status=status)


def bits(t):
    return t.view(torch.int16)


@pytest.mark.parametrize("maker", [workloads.heads_24_4, workloads.mixed_8x8])
def test_noalloc_matches_the_workspace_entry_point_twice(maker):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    # Another shape first, so the scratch holds another call's partials.
    without_allocation(workloads.split_sweep(3, 5, device="cuda", seed=30), status)
    for seed in (21, 22):  # two calls in a row, the second with other inputs
        case = maker(device="cuda", seed=seed)
        got = without_allocation(case, status)
        ref = with_workspace(case)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(bits(got), bits(ref)), f"seed {seed}: differs from k3da_attn_qknorm"
        assert_close(got, oracle_for(case), f"no-allocation seed {seed}")


def stride_case(stride, seed=23):
    return workloads.build_case(f"stride{stride}", R=8, B=8, Hq=24, Hkv=4, lens=[64] * 8, page_stride=stride,
                                used_per_row=1, num_pages=16, qknorm=True, seed=seed, device="cuda")


def test_noalloc_refuses_sizes_beyond_its_scratch():
    # The bound follows the chunk partials alone (the staging room that
    # k3da_workspace_bytes adds is optional here): page_stride 1279 runs,
    # 1280 and 2048 are refused.
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    case = stride_case(1279)
    got = without_allocation(case, status)
    ref = with_workspace(case)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(bits(got), bits(ref))
    for stride in (1280, 2048):
        with pytest.raises(k3da.K3daError):
            without_allocation(stride_case(stride), None)


def pinned(t):
    return t.cpu().contiguous().pin_memory()


@pytest.mark.parametrize("stride", [40, 1279])
def test_noalloc_with_host_resident_inputs(stride):
    """Inputs and output in pinned host memory: staged through the scratch
    where it has room (page_stride 40), read in place where it has not
    (1279, whose partials nearly fill it); bitwise the device-input call."""
    case = workloads.heads_24_4(device="cuda") if stride == 40 else stride_case(1279, seed=24)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full((case.T, case.Hq * case.D), float("nan"), dtype=torch.bfloat16).pin_memory()
    k3da.k3da_attn_qknorm_noalloc(out, pinned(case.qkv), case.pool, pinned(case.page_table),
                                  pinned(case.ctx_lens), pinned(case.positions), case.q_norm_w, case.k_norm_w,
                                  block_len=case.B, num_q_heads=case.Hq, num_kv_heads=case.Hkv, status=status)
    ref = with_workspace(case)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(bits(out), bits(ref).cpu())

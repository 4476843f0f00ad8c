"""The entry point that allocates nothing (k3da_attn_qknorm_noalloc).

Some callers cannot allocate device memory (host callbacks, real-time paths,
plugins whose host framework owns every allocation); for them the library
keeps a fixed scratch array on each GPU.  These tests call that entry point
through the C ABI and check its output against k3da_attn_qknorm (which takes
a caller-owned workspace) within the parity tolerance, on two calls in a row
with different inputs, and check that sizes beyond the array are refused.
Kept in the last test file so a run that stops at the first failure has
already run every other test."""
import numpy as np
import pytest
import torch

import speculative_decoding_drafter_k3_gb300 as k3da
from speculative_decoding_drafter_k3_gb300 import workloads
from common import ATOL, RTOL

pytestmark = pytest.mark.gpu


def with_workspace(case):
    out = torch.empty(case.T, case.Hq * case.D, dtype=torch.bfloat16, device="cuda")
    return k3da.k3da_attn_qknorm(out, case.qkv, case.pool, case.page_table, case.ctx_lens,
                                 case.positions, case.q_norm_w, case.k_norm_w, block_len=case.B,
                                 num_q_heads=case.Hq, num_kv_heads=case.Hkv,
                                 workspace=k3da.case_workspace(case))


def without_allocation(case, status):
    out = torch.empty(case.T, case.Hq * case.D, dtype=torch.bfloat16, device="cuda")
    return k3da.k3da_attn_qknorm_noalloc(out, case.qkv, case.pool, case.page_table, case.ctx_lens,
                                         case.positions, case.q_norm_w, case.k_norm_w,
                                         block_len=case.B, num_q_heads=case.Hq,
                                         num_kv_heads=case.Hkv, status=status)


def close(a, b):
    a = a.float().cpu().numpy()
    b = b.float().cpu().numpy()
    return np.isfinite(a).all() and bool((np.abs(a - b) <= ATOL + RTOL * np.abs(b)).all())


@pytest.mark.parametrize("maker", [workloads.heads_24_4, workloads.mixed_8x8])
def test_noalloc_matches_the_workspace_entry_point_twice(maker):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for seed in (21, 22):  # two calls in a row, the second with other inputs
        case = maker(device="cuda", seed=seed)
        ref = with_workspace(case)
        got = without_allocation(case, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert close(got, ref), f"seed {seed}: no-allocation output differs from k3da_attn_qknorm"


def test_noalloc_refuses_sizes_beyond_its_scratch():
    lib = k3da.load_library()
    cap = lib.k3da_noalloc_scratch_bytes()
    assert lib.k3da_workspace_bytes(8, 8, 24, 4, 1279) <= cap < lib.k3da_workspace_bytes(8, 8, 24, 4, 1280)
    assert lib.k3da_workspace_bytes(8, 8, 24, 4, 2048) > cap
    case = workloads.build_case("big", R=8, B=8, Hq=24, Hkv=4, lens=[64] * 8, page_stride=2048,
                                used_per_row=1, num_pages=16, qknorm=True, seed=23, device="cuda")
    with pytest.raises(k3da.K3daError):
        without_allocation(case, None)

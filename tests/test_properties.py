"""Properties the pages' tests ask of the op beyond parity (page "[None][feat]
Share Kimi K3 FP4 modeling and add NVFP4 support on SM103", NVIDIA/
TensorRT-LLM PR #20532, the drafter-attention commit's test list): no NaN,
the pool left byte-untouched, bit-identical reruns, isolated requests,
device-side range checks that flag and never fault, a poisoned workspace,
poisoned page-table tails and pool slots, and CUDA-graph replay with
rewritten lengths, page table, qkv and positions.  Reruns, the pool and
graph replay are checked on every workload of the op: the tiny plain call,
the 8x8 mixed-length and 24/4 strided cases, all eight request x token
splits and the long-context stress case."""
import dataclasses
import functools

import numpy as np
import pytest
import torch

import speculative_decoding_drafter_k3_gb300 as k3da
from oracle import units as ou
from speculative_decoding_drafter_k3_gb300 import workloads
from common import assert_close, oracle_for

pytestmark = pytest.mark.gpu

CONFIGS = dict([("tiny", workloads.tiny), ("mixed_8x8", workloads.mixed_8x8),
                ("heads_24_4", workloads.heads_24_4)]
               + [(f"split_{R}x{B}", functools.partial(workloads.split_sweep, R, B)) for R, B in workloads.SPLITS]
               + [("long_context", workloads.long_context)])


def fresh_out(case):
    return torch.empty(case.T, case.Hq * case.D, dtype=torch.bfloat16, device="cuda")


def whole_oracle(case):
    """The oracle on the whole call; the long-context case runs unit by unit
    on all host cores."""
    if case.context_tokens() > 100000:
        return ou.oracle_call(case)
    return oracle_for(case)


@pytest.mark.parametrize("config", sorted(CONFIGS))
def test_reruns_are_bit_identical_and_pool_untouched(config):
    case = CONFIGS[config](device="cuda")
    pool_before = case.pool.clone()
    ws = k3da.case_workspace(case)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    a = k3da.run_case(case, workspace=ws, status=status).clone()
    for _ in range(3):
        ws.fill_(0xFF)  # NaN-pattern workspace between calls
        b = k3da.run_case(case, workspace=ws, status=status)
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(case.pool.view(torch.int16), pool_before.view(torch.int16))
    assert torch.isfinite(a.float()).all()
    if config != "long_context":  # parity of the long-context case: test_parity
        assert_close(a, oracle_for(case), config)


def test_requests_are_isolated():
    case = workloads.mixed_8x8(device="cuda")
    base = k3da.run_case(case).clone()
    j = 3
    other = workloads.mixed_8x8(device="cuda")
    # Rewrite everything request j owns: its qkv rows, length, page row, positions.
    rows = slice(j * case.B, (j + 1) * case.B)
    case.qkv[rows] = torch.randn_like(case.qkv[rows].float()).to(torch.bfloat16)
    case.ctx_lens[j] = 1999
    case.page_table[j] = torch.flip(case.page_table[j], [0])
    case.positions[rows] += 7
    out = k3da.run_case(case)
    torch.cuda.synchronize()
    for r in range(case.R):
        sl = slice(r * case.B, (r + 1) * case.B)
        if r != j:
            assert torch.equal(out[sl].view(torch.int16), base[sl].view(torch.int16)), r
    assert_close(out, oracle_for(case), "isolation")
    del other


def test_poisoned_tails_and_stale_slots_are_never_used():
    case = workloads.build_case("poison", R=4, B=8, Hq=6, Hkv=1, lens=[65, 100, 0, 129],
                                page_stride=8, num_pages=64, qknorm=True, seed=70, device="cuda")
    ref = oracle_for(case)
    lens = case.lens_list()
    nan = torch.tensor(float("nan"), dtype=torch.bfloat16, device="cuda")
    used = set()
    for r, L in enumerate(lens):
        n = (L + 63) // 64
        case.page_table[r, n:] = -1 if r % 2 else 10 ** 6  # past the context: never read
        for p in range(n):
            page = int(case.page_table[r, p])
            used.add(page)
            if p == n - 1 and L % 64:
                case.pool[page, :, :, L % 64:, :] = nan  # stale slots after the context
    for page in range(case.num_pages):
        if page not in used:
            case.pool[page] = nan
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = k3da.run_case(case, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_close(out, ref, "poisoned")


def test_device_range_checks_flag_and_stay_finite():
    case = workloads.build_case("bad", R=2, B=4, Hq=6, Hkv=1, lens=[100, 50], page_stride=2,
                                num_pages=8, qknorm=True, seed=71, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    case.page_table[0, 1] = 8  # one past the pool
    out = k3da.run_case(case, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & k3da.STATUS_BAD_PAGE
    assert torch.isfinite(out.float()).all()
    case.page_table[0, 1] = 1
    case.ctx_lens[1] = 129  # beyond page_stride * 64
    status.zero_()
    out = k3da.run_case(case, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & k3da.STATUS_BAD_LENGTH
    assert torch.isfinite(out.float()).all()
    case.ctx_lens[1] = -5
    status.zero_()
    out = k3da.run_case(case, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & k3da.STATUS_BAD_LENGTH
    assert torch.isfinite(out.float()).all()


def test_host_side_refusals_raise():
    case = workloads.tiny(device="cuda")
    ws = k3da.case_workspace(case)
    with pytest.raises(k3da.K3daError):
        k3da.run_case(case, workspace=ws[:16])  # too small
    with pytest.raises(k3da.K3daError):
        k3da.k3da_attn(fresh_out(case), case.qkv, case.pool, case.page_table, case.ctx_lens,
                       block_len=case.B, num_q_heads=8, num_kv_heads=1, workspace=ws)


@pytest.mark.parametrize("config", sorted(CONFIGS))
def test_graph_replay_with_rewritten_inputs(config):
    """One call captured in a CUDA graph, then replayed after qkv, lengths,
    page table and positions (the fused variants) were rewritten in place:
    every replay equals an eager call bit for bit and the oracle element by
    element."""
    maker = CONFIGS[config]
    case = maker(device="cuda")
    ws = k3da.case_workspace(case)
    out = fresh_out(case)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    k3da.run_case(case, out=out, workspace=ws, status=status)  # first call outside capture
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        k3da.run_case(case, out=out, workspace=ws, status=status, stream=s)
    seeds = [11, 12] if config == "long_context" else [11, 12, 13]
    for seed in seeds:
        new = maker(device="cuda", seed=seed)
        case.qkv.copy_(new.qkv)
        case.ctx_lens.copy_(new.ctx_lens)
        case.page_table.copy_(new.page_table)
        if case.positions is not None:
            case.positions.copy_(new.positions)
        del new
        ws.fill_(0xFF)
        g.replay()
        torch.cuda.synchronize()
        replayed = out.clone()
        eager = k3da.run_case(case, workspace=ws, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(replayed.view(torch.int16), eager.view(torch.int16))
        if config != "long_context" or seed == seeds[-1]:
            assert_close(replayed, whole_oracle(case), f"{config} replay seed {seed}")


def test_a_stuck_wait_times_out_with_a_status_and_the_context_survives():
    """Failure detection without a fault: a wait on a barrier nothing
    completes gives up after its limit, raises TIMEOUT, releases the other
    warps, and later calls run normally."""
    import time
    lib = k3da.load_library()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    rc = lib.k3da_selftest_wait_timeout(ctypes_ptr(status), 5_000_000, None)  # 5 ms
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert rc == k3da.OK
    assert int(status.item()) == k3da.STATUS_TIMEOUT
    assert elapsed < 1.0, f"the other warps did not leave on the abort flag ({elapsed:.2f} s)"
    case = workloads.mixed_8x8(device="cuda")
    assert_close(k3da.run_case(case), oracle_for(case), "after a timed-out wait")


def ctypes_ptr(t):
    import ctypes
    return ctypes.c_void_p(t.data_ptr())


def test_calls_on_concurrent_streams_with_their_own_workspaces():
    """The library keeps no per-call state: calls in flight at the same time
    on different streams, each with its own workspace (one of them with
    host-resident inputs), give the bits of the same calls made one after
    the other."""
    makers = [workloads.mixed_8x8, workloads.heads_24_4, workloads.w6_8x6,
              functools.partial(workloads.split_sweep, 3, 5)]
    cases = [m(device="cuda") for m in makers]
    seq = [k3da.run_case(c).clone() for c in cases]
    torch.cuda.synchronize()
    host = cases[1]
    pinned = lambda t: t.cpu().contiguous().pin_memory()
    cases[1] = dataclasses.replace(host, qkv=pinned(host.qkv), page_table=pinned(host.page_table),
                                   ctx_lens=pinned(host.ctx_lens), positions=pinned(host.positions))
    streams = [torch.cuda.Stream() for _ in cases]
    wss = [k3da.case_workspace(c) for c in cases]
    outs = [fresh_out(c) for c in cases]
    status = [torch.zeros(1, dtype=torch.int32, device="cuda") for _ in cases]
    torch.cuda.synchronize()
    for _ in range(3):
        for c, s, w, o, st in zip(cases, streams, wss, outs, status):
            with torch.cuda.stream(s):
                o.fill_(float("nan"))
                k3da.run_case(c, out=o, workspace=w, status=st, stream=s)
        torch.cuda.synchronize()
        for o, ref, st in zip(outs, seq, status):
            assert int(st.item()) == 0
            assert torch.equal(o.view(torch.int16), ref.view(torch.int16))

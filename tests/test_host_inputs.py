"""Inputs and output in pinned host memory: a stage kernel copies qkv, the
positions and the lengths into the workspace across the host link, the split
pass reads the page table in place, and the combine writes the output to host
memory; no cudaMemcpy is involved.  The result must equal the call on
device-resident copies of the same tensors bit for bit (the same kernels run
on the same values), and a captured call must pick up host buffers rewritten
between replays."""
import dataclasses

import pytest
import torch

import speculative_decoding_drafter_k3_gb300 as k3da
from speculative_decoding_drafter_k3_gb300 import workloads
from common import assert_close, oracle_for

pytestmark = pytest.mark.gpu

CONFIGS = {
    "tiny": workloads.tiny,
    "mixed_8x8": workloads.mixed_8x8,
    "heads_24_4": workloads.heads_24_4,
    "w6_8x6": workloads.w6_8x6,
    "long_context_small": workloads.long_context_small,
    "long_context": workloads.long_context,
}


def pinned(t):
    return None if t is None else t.cpu().contiguous().pin_memory()


def host_side(case):
    """The case with qkv, page table, lengths and positions in pinned host
    memory (pool and norm weights stay on the GPU)."""
    return dataclasses.replace(case, qkv=pinned(case.qkv), page_table=pinned(case.page_table),
                               ctx_lens=pinned(case.ctx_lens), positions=pinned(case.positions))


def host_out(case):
    return torch.full((case.T, case.Hq * case.D), float("nan"), dtype=torch.bfloat16).pin_memory()


@pytest.mark.parametrize("config", list(CONFIGS))
def test_host_inputs_equal_device_inputs_bit_for_bit(config):
    case = CONFIGS[config](device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dev_out = k3da.run_case(case, status=status)
    hcase = host_side(case)
    out = host_out(case)
    k3da.run_case(hcase, out=out, workspace=k3da.case_workspace(case), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(out.view(torch.int16), dev_out.cpu().view(torch.int16))
    if config in ("tiny", "mixed_8x8"):
        assert_close(out.cuda(), oracle_for(case), f"{config} from host memory")


@pytest.mark.parametrize("which", ["qkv", "page_table", "ctx_lens", "positions", "out"])
def test_each_tensor_alone_in_host_memory(which):
    """One tensor host-resident, the rest on the device (qkv, positions or
    lengths alone still take the staged path); int64 positions, strided
    page-table rows."""
    case = workloads.heads_24_4(device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref = k3da.run_case(case, status=status)
    c = case if which == "out" else dataclasses.replace(case, **{which: pinned(getattr(case, which))})
    out = host_out(case) if which == "out" else torch.empty_like(ref)
    k3da.run_case(c, out=out, workspace=k3da.case_workspace(case), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(out.cpu().view(torch.int16), ref.cpu().view(torch.int16))


def test_graph_replay_reads_rewritten_host_buffers():
    case = workloads.mixed_8x8(device="cuda")
    hcase = host_side(case)
    out = host_out(case)
    ws = k3da.case_workspace(case)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    k3da.run_case(hcase, out=out, workspace=ws, status=status)  # first call outside capture
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        k3da.run_case(hcase, out=out, workspace=ws, status=status, stream=s)
    for seed in (21, 22):
        new = workloads.mixed_8x8(device="cpu", seed=seed)
        hcase.qkv.copy_(new.qkv)
        hcase.page_table.copy_(new.page_table)
        hcase.ctx_lens.copy_(new.ctx_lens)
        hcase.positions.copy_(new.positions)
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        eager = k3da.run_case(dataclasses.replace(case, qkv=new.qkv.cuda(), page_table=new.page_table.cuda(),
                                                  ctx_lens=new.ctx_lens.cuda(), positions=new.positions.cuda()),
                              status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(out.view(torch.int16), eager.cpu().view(torch.int16))


def test_pool_workspace_and_unpinned_inputs_are_refused():
    case = workloads.tiny(device="cuda")
    hcase = host_side(case)
    out = host_out(case)
    ws = k3da.case_workspace(case)
    kw = dict(block_len=case.B, num_q_heads=case.Hq, num_kv_heads=case.Hkv)
    with pytest.raises(k3da.K3daError):  # the pool is device memory only
        k3da.k3da_attn(out, hcase.qkv, pinned(case.pool), hcase.page_table, hcase.ctx_lens, workspace=ws, **kw)
    with pytest.raises(k3da.K3daError):  # so is the workspace
        k3da.k3da_attn(out, hcase.qkv, case.pool, hcase.page_table, hcase.ctx_lens,
                       workspace=pinned(ws), **kw)
    with pytest.raises(k3da.K3daError):  # pageable host memory is not addressed by the kernels
        k3da.k3da_attn(out, case.qkv.cpu(), case.pool, hcase.page_table, hcase.ctx_lens, workspace=ws, **kw)

"""Parity of the standalone q/k RMSNorm + NeoX RoPE call (k3da_qk_norm_rope)
with the fp64 oracle, plus its in-place contract (GPU).

Tolerance, from the arithmetic: the kernel widens bf16 inputs exactly,
normalises and rotates in fp32 (angles reduced exactly in integer turns,
accurate sincospif) and rounds each result to bf16 once, so
|gpu - oracle| <= 2^-9 |oracle| from the final rounding plus ~1e-6 from fp32
on values of magnitude ~4; the test allows 2^-8 |oracle| + 1e-4."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_drafter_k3_gb300 as k3da

pytestmark = pytest.mark.gpu
D = 64
RTOL = 2.0 ** -8
ATOL = 1e-4


def make(T, Hq, Hkv, pos_dtype, seed, pos_hi=1 << 17):
    g = torch.Generator().manual_seed(seed)
    qkv = torch.randn(T, (Hq + 2 * Hkv) * D, generator=g).to(torch.bfloat16)
    qw = (1 + 0.1 * torch.randn(D, generator=g)).to(torch.bfloat16)
    kw = (1 + 0.1 * torch.randn(D, generator=g)).to(torch.bfloat16)
    pos = torch.randint(0, pos_hi, (T,), generator=g).to(pos_dtype)
    return qkv, qw, kw, pos


def run(qkv, qw, kw, pos, Hq, Hkv):
    dev = [t.cuda() for t in (qkv, qw, kw, pos)]
    k3da.k3da_qk_norm_rope(dev[0], dev[3], dev[1], dev[2], num_q_heads=Hq, num_kv_heads=Hkv)
    torch.cuda.synchronize()
    return dev[0].cpu()


@pytest.mark.parametrize("T", [1, 7, 64, 333])
@pytest.mark.parametrize("Hq,Hkv", [(6, 1), (24, 4)])
@pytest.mark.parametrize("pos_dtype", [torch.int32, torch.int64])
def test_matches_oracle(T, Hq, Hkv, pos_dtype):
    qkv, qw, kw, pos = make(T, Hq, Hkv, pos_dtype, seed=T * 31 + Hq)
    got = run(qkv, qw, kw, pos, Hq, Hkv).double().numpy()
    ref = oracle.qk_norm_rope(qkv, pos, qw, kw, num_q_heads=Hq, num_kv_heads=Hkv)
    err = np.abs(got - ref)
    assert np.isfinite(got).all()
    assert (err <= ATOL + RTOL * np.abs(ref)).all(), f"max err {err.max():.3e}"
    # Value heads are not touched: bit for bit the input.
    v0 = (Hq + Hkv) * D
    assert torch.equal(run(qkv, qw, kw, pos, Hq, Hkv)[:, v0:].view(torch.int16), qkv[:, v0:].view(torch.int16))


def test_large_positions_keep_the_angle_exact():
    qkv, qw, kw, pos = make(16, 6, 1, torch.int64, seed=5, pos_hi=1 << 40)
    got = run(qkv, qw, kw, pos, 6, 1).double().numpy()
    ref = oracle.qk_norm_rope(qkv, pos, qw, kw, num_q_heads=6, num_kv_heads=1)
    assert (np.abs(got - ref) <= ATOL + RTOL * np.abs(ref)).all()


def test_reruns_bitwise_and_graph_replay_with_new_positions():
    Hq, Hkv, T = 24, 4, 64
    qkv, qw, kw, pos = make(T, Hq, Hkv, torch.int64, seed=9)
    dq, dw, dk, dp = qkv.cuda(), qw.cuda(), kw.cuda(), pos.cuda()
    work = dq.clone()
    k3da.k3da_qk_norm_rope(work, dp, dw, dk, num_q_heads=Hq, num_kv_heads=Hkv)
    first = work.clone()
    work.copy_(dq)
    k3da.k3da_qk_norm_rope(work, dp, dw, dk, num_q_heads=Hq, num_kv_heads=Hkv)
    assert torch.equal(first.view(torch.int16), work.view(torch.int16))
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        work.copy_(dq)
        torch.cuda.synchronize()
        with torch.cuda.graph(graph, stream=s):
            k3da.k3da_qk_norm_rope(work, dp, dw, dk, num_q_heads=Hq, num_kv_heads=Hkv, stream=s)
    new_pos = pos + 1000
    dp.copy_(new_pos.cuda())
    work.copy_(dq)
    graph.replay()
    torch.cuda.synchronize()
    ref = oracle.qk_norm_rope(qkv, new_pos, qw, kw, num_q_heads=Hq, num_kv_heads=Hkv)
    got = work.cpu().double().numpy()
    assert (np.abs(got - ref) <= ATOL + RTOL * np.abs(ref)).all()


@pytest.mark.parametrize("config,yarn", [("mixed_8x8", False), ("heads_24_4", False), ("heads_24_4", True),
                                         ("w6_8x6", True)])
def test_norm_rope_then_plain_attention_gives_the_fused_bits(config, yarn):
    """This call applies to the block exactly what the fused attention's
    prologue applies (the same operations, rounded the same way), so
    normalising the block with it and then calling the plain attention must
    give the fused attention's output bit for bit (and both match the
    oracle)."""
    from speculative_decoding_drafter_k3_gb300 import workloads
    from common import assert_close, oracle_for
    case = getattr(workloads, config)(device="cuda")
    y = k3da.Yarn.of(4.0, 4096.0) if yarn else None
    fused = k3da.run_case(case, yarn=y).clone()
    qkv = case.qkv.clone()
    k3da.k3da_qk_norm_rope(qkv, case.positions, case.q_norm_w, case.k_norm_w, num_q_heads=case.Hq,
                           num_kv_heads=case.Hkv, yarn=y)
    ws = k3da.case_workspace(case)
    out = torch.empty_like(fused)
    k3da.k3da_attn(out, qkv, case.pool, case.page_table, case.ctx_lens, block_len=case.B,
                   num_q_heads=case.Hq, num_kv_heads=case.Hkv, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), fused.view(torch.int16))
    if not yarn:
        assert_close(out, oracle_for(case), f"{config}: norm_rope then plain attention")

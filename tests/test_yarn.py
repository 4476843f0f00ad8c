"""YaRN RoPE in the fused attention and in the standalone norm+RoPE cell
against the fp64 oracle (GPU).  The drafter's setting on the pages is "YaRN
4.0"; the other parameters are the YaRN paper's (beta_fast 32, beta_slow 1,
mscale 0.1 ln(s) + 1) with an original context of 4096 positions.  The GPU
calls pass mscale 0, so the library forms the paper's default itself; the
oracle is given that default explicitly.  Tolerances are those of the plain paths: 2e-2 + 2e-2 |ref| for
the attention output, 2^-8 |ref| + 1e-4 for the cell."""
import math

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_drafter_k3_gb300 as k3da
from speculative_decoding_drafter_k3_gb300 import workloads
from common import assert_close

pytestmark = pytest.mark.gpu
YARN = k3da.Yarn.of(4.0, 4096.0, 32.0, 1.0)  # mscale 0: the library's default
PAPER_MSCALE = 0.1 * math.log(4.0) + 1.0
YARN_FOR_ORACLE = dict(YARN.as_dict(), mscale=PAPER_MSCALE)


def oracle_yarn(case, yarn_dict):
    return oracle.attn(case.qkv, case.pool, case.page_table, case.ctx_lens, num_requests=case.R,
                       block_len=case.B, num_q_heads=case.Hq, num_kv_heads=case.Hkv, scale=case.scale,
                       qknorm=True, positions=case.positions, q_norm_w=case.q_norm_w, k_norm_w=case.k_norm_w,
                       eps=case.eps, rope_base=case.rope_base, yarn=yarn_dict)


@pytest.mark.parametrize("maker", [workloads.mixed_8x8, workloads.heads_24_4, workloads.w6_8x6])
def test_attention_with_yarn_matches_oracle(maker):
    case = maker(device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = k3da.run_case(case, status=status, yarn=YARN)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_close(out, oracle_yarn(case, YARN_FOR_ORACLE), case.name + " yarn")
    # The rescaling changes the result (it is not silently ignored).
    plain = k3da.run_case(case)
    assert not torch.equal(out.view(torch.int16), plain.view(torch.int16))


def test_yarn_default_mscale_is_the_papers_value_rounded_to_fp32():
    """mscale 0 makes the library use 0.1 ln(factor) + 1 rounded once to
    fp32: bitwise the call that passes that fp32 value explicitly."""
    case = workloads.mixed_8x8(device="cuda")
    default = k3da.run_case(case, yarn=YARN).clone()
    explicit = k3da.Yarn.of(4.0, 4096.0, 32.0, 1.0, mscale=float(np.float32(PAPER_MSCALE)))
    assert explicit.mscale == np.float32(PAPER_MSCALE)
    same = k3da.run_case(case, yarn=explicit)
    assert torch.equal(default.view(torch.int16), same.view(torch.int16))


def test_yarn_factor_one_is_bitwise_the_plain_call():
    case = workloads.heads_24_4(device="cuda")
    plain = k3da.run_case(case).clone()
    same = k3da.run_case(case, yarn=k3da.Yarn(1.0, 4096.0, 32.0, 1.0, 1.0))
    assert torch.equal(plain.view(torch.int16), same.view(torch.int16))


@pytest.mark.parametrize("Hq,Hkv", [(6, 1), (24, 4)])
def test_norm_rope_cell_with_yarn_matches_oracle(Hq, Hkv):
    g = torch.Generator().manual_seed(77 + Hq)
    T, D = 64, 64
    qkv = torch.randn(T, (Hq + 2 * Hkv) * D, generator=g).to(torch.bfloat16)
    qw = (1 + 0.1 * torch.randn(D, generator=g)).to(torch.bfloat16)
    kw = (1 + 0.1 * torch.randn(D, generator=g)).to(torch.bfloat16)
    pos = torch.randint(0, 1 << 17, (T,), generator=g, dtype=torch.int64)
    dev = qkv.cuda()
    k3da.k3da_qk_norm_rope(dev, pos.cuda(), qw.cuda(), kw.cuda(), num_q_heads=Hq, num_kv_heads=Hkv, yarn=YARN)
    torch.cuda.synchronize()
    got = dev.cpu().double().numpy()
    ref = oracle.qk_norm_rope(qkv, pos, qw, kw, num_q_heads=Hq, num_kv_heads=Hkv, yarn=YARN_FOR_ORACLE)
    assert (np.abs(got - ref) <= 1e-4 + 2.0 ** -8 * np.abs(ref)).all()

"""Parity of the CUDA path with the fp64 oracle, element by element, on the
five workloads of the drafter block attention (6/1 and 24/4 heads, every
request x token split, context lengths 0..2041 and 16k..128k, dense and
strided page-table rows, int32 and int64 positions), plus edge cases.
Tolerance: |gpu - oracle| <= 2e-2 + 2e-2 |oracle| on the bf16 output."""
import dataclasses

import numpy as np
import pytest
import torch

import speculative_decoding_drafter_k3_gb300 as k3da
from oracle import units as ou
from speculative_decoding_drafter_k3_gb300 import workloads
from common import assert_close, oracle_for

pytestmark = pytest.mark.gpu


def run(case, **kw):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = k3da.run_case(case, status=status, **kw)
    torch.cuda.synchronize()
    return out, int(status.item())


def check(case):
    out, st = run(case)
    assert st == 0, f"{case.name}: device status {st}"
    return assert_close(out, oracle_for(case), case.name)


def test_tiny_plain_variant():
    check(workloads.tiny(device="cuda"))


def test_mixed_lengths_8x8_6_1_int32():
    check(workloads.mixed_8x8(device="cuda"))


def test_heads_24_4_strided_rows_int64():
    check(workloads.heads_24_4(device="cuda"))


@pytest.mark.parametrize("R,B", workloads.SPLITS)
def test_split_sweep(R, B):
    check(workloads.split_sweep(R, B, device="cuda"))


@pytest.mark.parametrize("R,B", [(8, 8), (3, 5)])
def test_split_sweep_plain_variant(R, B):
    case = workloads.split_sweep(R, B, device="cuda", seed=50)
    case.qknorm = False
    check(case)


@pytest.mark.parametrize("lens", [
    [0] * 8,                          # block-only attention everywhere
    [1, 63, 64, 65, 127, 128, 129, 2048],  # page boundaries, full row
    [2048] * 8,                       # every page-table entry used
])
@pytest.mark.parametrize("Hq,Hkv", [(6, 1), (24, 4)])
def test_edge_lengths(lens, Hq, Hkv):
    case = workloads.build_case("edge", R=8, B=8, Hq=Hq, Hkv=Hkv, lens=lens, page_stride=32,
                                num_pages=512, qknorm=True, pos_dtype=torch.int64, seed=60,
                                device="cuda")
    check(case)


@pytest.mark.parametrize("R,B", [(1, 1), (1, 8), (3, 5), (5, 3), (8, 1)])
@pytest.mark.parametrize("qknorm,pos_dtype", [(True, torch.int32), (True, torch.int64), (False, torch.int32)])
def test_heads_24_4_request_token_splits(R, B, qknorm, pos_dtype):
    """The 24/4 layout over request x token splits, both position types and
    the plain variant; lengths from the split sweep's set plus a 10k context."""
    g = torch.Generator().manual_seed(700 + 10 * R + B)
    choices = workloads.SWEEP_LENGTHS + [10000]
    lens = [choices[int(i)] for i in torch.randint(0, len(choices), (R,), generator=g)]
    case = workloads.build_case(f"h24_{R}x{B}", R=R, B=B, Hq=24, Hkv=4, lens=lens, page_stride=160,
                                num_pages=R * 160, qknorm=qknorm, pos_dtype=pos_dtype, seed=71 + R * B,
                                device="cuda")
    check(case)


def test_lengths_at_full_size_chunk_edges():
    """8 requests x 24/4 heads (32 units: chunks of 32 pages once a unit has
    more than ~500 items): contexts whose page counts sit on and next to a
    chunk edge, a partial last page, one page, and no context."""
    lens = [639 * 64, 640 * 64, 640 * 64 + 1, 513 * 64 - 5, 512 * 64, 511 * 64 + 63, 64, 0]
    case = workloads.build_case("chunk_edges", R=8, B=8, Hq=24, Hkv=4, lens=lens, page_stride=641,
                                num_pages=8 * 641, qknorm=True, pos_dtype=torch.int64, seed=64,
                                device="cuda")
    check(case)


def test_single_token_single_request():
    case = workloads.build_case("1x1", R=1, B=1, Hq=24, Hkv=4, lens=[777], page_stride=13,
                                num_pages=40, qknorm=True, seed=61, device="cuda")
    check(case)


def test_large_positions_keep_rope_angles_exact():
    # Positions near 131k: the RoPE angle must not lose precision.
    case = workloads.build_case("bigpos", R=2, B=8, Hq=6, Hkv=1, lens=[100, 5], page_stride=4,
                                num_pages=16, qknorm=True, pos_dtype=torch.int64, seed=62,
                                device="cuda")
    case.positions = case.positions + 131000
    check(case)


def _rescale_case(R, Hq, Hkv, L, seed):
    """A plain-variant case whose row maximum jumps once per 8 pages.

    Every query row is 1/8 (all dims).  The keys of pages 5, 13, 21, ... of
    each context are 6 (all dims) and all other keys, block keys included,
    are 0.  So those pages score 6 * 1.4427 = 8.7 log2 units above the rest,
    more than the 8 past which the split pass moves a row's exponent base and
    rescales its O.  Whatever power-of-two chunk size of 4 items or more a
    unit gets, such a page sits inside a chunk whose first item scores 0, so
    every such chunk rescales once, at a position that differs between
    chunks (and so at every S/P buffer index).  Values are +1 on the high
    pages and -1 elsewhere (plus 0.1 N(0, 1)).  The output is then about
    +0.98; an O or l left unscaled moves it far from that."""
    n = L // 64
    case = workloads.build_case(f"rescale_{R}x8_{Hq}/{Hkv}_L{L}", R=R, B=8, Hq=Hq, Hkv=Hkv, lens=[L] * R,
                                page_stride=n, num_pages=R * n, qknorm=False, seed=seed, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(seed)
    qkv = case.qkv.view(case.T, Hq + 2 * Hkv, 64)
    qkv[:, :Hq] = 0.125
    qkv[:, Hq:Hq + Hkv] = 0.0
    qkv[:, Hq + Hkv:] = (-1.0 + 0.1 * torch.randn(qkv[:, Hq + Hkv:].shape, generator=g, device="cuda")).to(torch.bfloat16)
    high = torch.zeros(R * n, dtype=torch.bool, device="cuda")
    pages = case.page_table[:, :n].long()
    high[pages[:, 5::8].reshape(-1)] = True
    pool = case.pool
    pool[:, 0] = 0.0
    pool[high, 0] = 6.0
    noise = 0.1 * torch.randn(pool[:, 1].shape, generator=g, device="cuda")
    sign = torch.where(high, 1.0, -1.0).view(-1, 1, 1, 1)
    pool[:, 1] = (sign + noise).to(torch.bfloat16)
    return case


@pytest.mark.parametrize("R,Hq,Hkv,L", [(2, 6, 1, 65536), (8, 24, 4, 40960), (1, 6, 1, 8192)])
def test_rows_whose_maximum_jumps_mid_chunk(R, Hq, Hkv, L):
    case = _rescale_case(R, Hq, Hkv, L, seed=90 + R)
    ref = oracle_for(case)
    assert 0.9 < float(np.median(ref)) < 1.0  # the high pages dominate, the low ones still count
    out, st = run(case)
    assert st == 0
    assert_close(out, ref, case.name)


def test_huge_page_stride_short_contexts():
    """page_stride 200,000 (each unit gets 6,251 workspace slots, so slot
    indices and the combine's reads reach ~12,500 slots deep) with short
    contexts; the page-table rows are poison past their first 100 entries."""
    case = workloads.build_case("stride200k", R=2, B=8, Hq=6, Hkv=1, lens=[5000, 64], page_stride=200000,
                                used_per_row=100, num_pages=200, qknorm=True, seed=95, device="cuda")
    check(case)


def test_positions_beyond_32_bits():
    """int64 positions near 2^33 and 2^40 in the fused attention: the angle
    is reduced exactly as a fraction of a turn in 64-bit integers."""
    for base_pos, seed in ((2 ** 33 + 12345, 96), (2 ** 40 - 77, 97)):
        case = workloads.build_case("bigpos64", R=2, B=8, Hq=24, Hkv=4, lens=[300, 2041], page_stride=32,
                                    num_pages=64, qknorm=True, pos_dtype=torch.int64, seed=seed, device="cuda")
        case.positions = case.positions + base_pos
        check(case)


@pytest.mark.parametrize("rope_base,eps", [(500000.0, 1e-6), (1000.0, 1e-3)])
def test_other_rope_base_and_eps(rope_base, eps):
    case = workloads.build_case("base_eps", R=4, B=8, Hq=6, Hkv=1, lens=[2041, 700, 64, 0], page_stride=32,
                                num_pages=128, qknorm=True, seed=98, device="cuda")
    case = dataclasses.replace(case, rope_base=rope_base, eps=eps)
    check(case)


@pytest.mark.parametrize("scale,qknorm", [(0.2, True), (0.05, False)])
def test_other_softmax_scales(scale, qknorm):
    case = workloads.build_case("scale", R=3, B=5, Hq=24, Hkv=4, lens=[1500, 65, 2041], page_stride=32,
                                num_pages=96, qknorm=qknorm, seed=99, device="cuda")
    check(dataclasses.replace(case, scale=scale))


def test_production_block_width_w6_8x6():
    check(workloads.w6_8x6(device="cuda"))


@pytest.mark.parametrize("maker", [workloads.single_w6, workloads.single_w6_long])
def test_single_request_w6(maker):
    check(maker(device="cuda"))


def test_long_context_every_request():
    """The long-context workload at full size (20k-page pool, 16k..128k
    contexts, 24/4 heads), in the launch configuration the benchmark uses,
    against the oracle on every request: the call's 32 (request, kv head)
    units run through the oracle one by one on all host cores."""
    case = workloads.long_context(device="cuda")
    out, st = run(case)
    assert st == 0
    ref = ou.oracle_call(case)
    assert not np.isnan(ref).any()
    assert_close(out, ref, "long_context")


BALANCED_LENS = [131072, 2041, 0, 64, 65536, 16385, 1, 100000]


def _balanced_pair():
    """Two calls that differ only in request 2's context (0 tokens, then
    5000): same pool, qkv, norm weights and page-table rows (each a slice of
    one page permutation, sized for the longer of the two lengths; entries
    past a context are never read)."""
    lens1 = list(BALANCED_LENS)
    lens2 = list(BALANCED_LENS)
    lens2[2] = 5000
    need = [(max(a, b) + 63) // 64 for a, b in zip(lens1, lens2)]
    g = torch.Generator().manual_seed(66)
    perm = torch.randperm(sum(need) + 16, generator=g).to(torch.int32)
    case = workloads.build_case("balanced_mixed", R=8, B=8, Hq=24, Hkv=4, lens=[0] * 8, page_stride=2048,
                                num_pages=sum(need) + 16, used_per_row=1, qknorm=True,
                                pos_dtype=torch.int64, seed=66, device="cuda")
    pt = torch.full((8, 2048), -1, dtype=torch.int32)
    off = 0
    for r, n in enumerate(need):
        pt[r, :n] = perm[off:off + n]
        off += n
    case.page_table.copy_(pt)
    cases = []
    for lens in (lens1, lens2):
        c = dataclasses.replace(case, ctx_lens=torch.tensor(lens, dtype=torch.int32, device="cuda"),
                                positions=torch.tensor([L + i for L in lens for i in range(8)],
                                                       dtype=torch.int64, device="cuda"))
        cases.append(c)
    return cases


def test_balanced_assignment_with_mixed_chunk_sizes():
    """Contexts long enough for the balanced assignment (every CTA holds
    several 32-page chunks, so the work is cut on the nominal line of chunk
    sizes) mixed with short ones (3- and 1-item chunks): every request
    matches the oracle, and changing one request's length, which moves
    every CTA's share of the work, leaves the other requests' rows bitwise
    unchanged."""
    case1, case2 = _balanced_pair()
    out1, st1 = run(case1)
    out1 = out1.clone()
    assert st1 == 0
    assert_close(out1, ou.oracle_call(case1), "balanced_mixed")
    out2, st2 = run(case2)
    assert st2 == 0
    for r in range(8):
        if r != 2:
            sl = slice(r * 8, (r + 1) * 8)
            assert torch.equal(out1[sl].view(torch.int16), out2[sl].view(torch.int16)), r
    ref2 = ou.oracle_call(case2, requests=[2])
    assert_close(out2[16:24], ref2[16:24], "balanced_mixed r2")

"""Parity of the CUDA path with the fp64 oracle, element by element, on the
five workloads of the drafter block attention (6/1 and 24/4 heads, every
request x token split, context lengths 0..2041 and 16k..128k, dense and
strided page-table rows, int32 and int64 positions), plus edge cases.
Tolerance: |gpu - oracle| <= 2e-2 + 2e-2 |oracle| on the bf16 output."""
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

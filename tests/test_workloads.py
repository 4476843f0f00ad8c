"""The seeded synthetic inputs have the shapes, distributions and structure the
workloads promise (CPU only): lengths in range, page-table rows that are
disjoint slices of one permutation with poisoned tails, positions = context
length + token index, deterministic draws, and the algorithmic byte count the
benchmark reports.  Only small workloads are drawn in full here; the
long-context one is checked through its lengths and byte count."""
import pytest
import torch

from speculative_decoding_drafter_k3_gb300 import workloads

SMALL = ["tiny", "mixed_8x8", "heads_24_4", "w6_8x6", "single_w6"]


@pytest.mark.parametrize("name", SMALL)
def test_shapes_and_layouts(name):
    c = workloads.WORKLOADS[name]()
    T = c.R * c.B
    assert tuple(c.qkv.shape) == (T, (c.Hq + 2 * c.Hkv) * 64) and c.qkv.dtype == torch.bfloat16
    assert tuple(c.pool.shape) == (c.num_pages, 2, c.Hkv, 64, 64) and c.pool.dtype == torch.bfloat16
    assert tuple(c.page_table.shape) == (c.R, c.page_stride) and c.page_table.dtype == torch.int32
    assert tuple(c.ctx_lens.shape) == (c.R,) and c.ctx_lens.dtype == torch.int32
    assert (c.Hq, c.Hkv) in [(6, 1), (24, 4)] and 1 <= c.B <= 8 and 1 <= c.R <= 8
    if c.qknorm:
        assert c.positions.dtype == c.pos_dtype and c.positions.numel() == T
        assert c.q_norm_w.shape == (64,) and c.k_norm_w.shape == (64,)


@pytest.mark.parametrize("name", SMALL)
def test_page_tables_are_disjoint_permutation_slices_with_poisoned_tails(name):
    c = workloads.WORKLOADS[name]()
    seen = set()
    for r, L in enumerate(c.lens_list()):
        assert 0 <= L <= c.page_stride * 64
        row = c.page_table[r].tolist()
        used = [p for p in row if p != workloads.POISON_PAGE]
        assert used == row[:len(used)], "poison only after the used entries"
        assert len(used) * 64 >= L
        assert all(0 <= p < c.num_pages for p in used)
        assert not (seen & set(used)), "rows never share a page"
        seen |= set(used)


@pytest.mark.parametrize("name", [n for n in SMALL if workloads.WORKLOADS[n]().qknorm])
def test_positions_continue_each_context(name):
    c = workloads.WORKLOADS[name]()
    lens = c.lens_list()
    want = [lens[r] + i for r in range(c.R) for i in range(c.B)]
    assert c.positions.tolist() == want


def test_length_distributions():
    assert workloads.tiny().lens_list() == [100]
    assert all(L == 2041 for L in workloads.heads_24_4().lens_list())
    for seed in range(3):
        assert all(0 <= L <= 2041 for L in workloads.mixed_8x8(seed=seed).lens_list())
    for R, B in workloads.SPLITS:
        assert all(L in workloads.SWEEP_LENGTHS for L in workloads.split_sweep(R, B).lens_list())
    g = workloads._gen(4 + 307, "cpu")
    long_lens = torch.randint(16384, 131072 + 1, (8,), generator=g).tolist()
    assert all(16384 <= L <= 131072 for L in long_lens)


def test_draws_are_deterministic_per_seed():
    a, b = workloads.mixed_8x8(seed=9), workloads.mixed_8x8(seed=9)
    assert torch.equal(a.qkv.view(torch.int16), b.qkv.view(torch.int16))
    assert torch.equal(a.page_table, b.page_table) and a.lens_list() == b.lens_list()
    c = workloads.mixed_8x8(seed=10)
    assert not torch.equal(a.qkv.view(torch.int16), c.qkv.view(torch.int16))


def test_algorithmic_bytes_count_each_input_once():
    c = workloads.tiny()
    kv = 100 * 1 * 2 * 64 * 2
    qkv = 4 * 8 * 64 * 2
    out = 4 * 6 * 64 * 2
    pages = 2 * 4
    assert c.algorithmic_bytes() == kv + qkv + out + pages + 1 * 4
    m = workloads.mixed_8x8()
    extra = m.T * 4 + 2 * 64 * 2  # int32 positions and the two weight vectors
    lens = m.lens_list()
    assert m.algorithmic_bytes() == (sum(lens) * 256 + m.T * 8 * 128 + m.T * 6 * 128
                                     + sum((L + 63) // 64 for L in lens) * 4 + 8 * 4 + extra)


def test_request_view_is_the_independent_sub_problem():
    c = workloads.mixed_8x8()
    s = c.request(3)
    assert s.R == 1 and s.lens_list() == [c.lens_list()[3]]
    assert torch.equal(s.qkv.view(torch.int16), c.qkv[3 * c.B:4 * c.B].view(torch.int16))
    assert torch.equal(s.page_table, c.page_table[3:4])
    assert s.positions.tolist() == c.positions[3 * c.B:4 * c.B].tolist()

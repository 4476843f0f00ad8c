"""Seeded synthetic inputs of the drafter block attention.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic, so both the CUDA path and the fp64 oracle can be fed from
it.  The shapes and distributions follow the op as the page "[None][feat]
Share Kimi K3 FP4 modeling and add NVFP4 support on SM103" (NVIDIA/TensorRT-LLM
PR #20532) describes it: up to 8 requests with draft blocks of up to 8 tokens,
6/1 or 24/4 query/KV heads, head_dim 64, HND pages of 64 tokens, context
lengths 0..2041, dense or strided page-table rows with padded page strides,
int32 or int64 positions, eps 1e-5, RoPE base 10000.

Layouts (all row-major):
  qkv         [T, (Hq + 2*Hkv) * 64] bf16, T = R*B, row r*B + i = request r,
              token i; q heads, then k heads, then v heads
  pool        [num_pages, 2, Hkv, 64, 64] bf16 (K = 0, V = 1)
  page_table  [R, page_stride] int32
  ctx_lens    [R] int32
  positions   [T] int32 or int64, ctx_len + i
  q_norm_w,
  k_norm_w    [64] bf16, 1 + 0.1 * N(0, 1)
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence

import torch

HEAD_DIM = 64
PAGE_SIZE = 64
POISON_PAGE = -1


@dataclasses.dataclass
class Case:
    name: str
    R: int
    B: int
    Hq: int
    Hkv: int
    page_stride: int
    num_pages: int
    qknorm: bool
    pos_dtype: torch.dtype
    qkv: torch.Tensor
    pool: torch.Tensor
    page_table: torch.Tensor
    ctx_lens: torch.Tensor
    positions: Optional[torch.Tensor]
    q_norm_w: Optional[torch.Tensor]
    k_norm_w: Optional[torch.Tensor]
    scale: float = 0.125
    eps: float = 1e-5
    rope_base: float = 10000.0
    D: int = HEAD_DIM
    P: int = PAGE_SIZE

    @property
    def T(self) -> int:
        return self.R * self.B

    def lens_list(self) -> list:
        return [int(x) for x in self.ctx_lens.cpu().tolist()]

    def context_tokens(self) -> int:
        return sum(self.lens_list())

    def algorithmic_bytes(self) -> int:
        """Bytes the op must move once: context K/V, qkv, out, the page ids
        it reads, lengths, positions and norm weights."""
        lens = self.lens_list()
        kv = sum(lens) * self.Hkv * 2 * self.D * 2
        qkv = self.T * (self.Hq + 2 * self.Hkv) * self.D * 2
        out = self.T * self.Hq * self.D * 2
        pt = sum((L + self.P - 1) // self.P for L in lens) * 4
        extra = self.R * 4
        if self.qknorm:
            extra += self.T * (8 if self.pos_dtype == torch.int64 else 4) + 2 * self.D * 2
        return kv + qkv + out + pt + extra

    def to(self, device) -> "Case":
        def mv(t):
            return None if t is None else t.to(device)

        return dataclasses.replace(
            self, qkv=mv(self.qkv), pool=mv(self.pool), page_table=mv(self.page_table),
            ctx_lens=mv(self.ctx_lens), positions=mv(self.positions),
            q_norm_w=mv(self.q_norm_w), k_norm_w=mv(self.k_norm_w))

    def request(self, r: int) -> "Case":
        """The sub-problem of request r alone (requests are independent)."""
        rows = slice(r * self.B, (r + 1) * self.B)
        return dataclasses.replace(
            self, name=f"{self.name}[r{r}]", R=1, qkv=self.qkv[rows],
            page_table=self.page_table[r:r + 1], ctx_lens=self.ctx_lens[r:r + 1],
            positions=None if self.positions is None else self.positions[rows])


def _normal_bf16(shape, gen: torch.Generator, device) -> torch.Tensor:
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def build_case(name: str, *, R: int, B: int, Hq: int, Hkv: int, lens: Sequence[int],
               page_stride: int, num_pages: int, qknorm: bool, pos_dtype=torch.int32,
               used_per_row: Optional[int] = None, seed: int = 0, device="cpu") -> Case:
    """Draw one case.

    Page-table row r holds a consecutive slice of one random permutation of
    the pool's pages (``used_per_row`` entries, default ``page_stride``); the
    rest of the row is POISON_PAGE.  qkv and the pool are N(0, 1) bf16, drawn
    on ``device`` from a generator seeded with ``seed``; the small tensors are
    drawn on the CPU from the same seed.
    """
    assert len(lens) == R
    used = page_stride if used_per_row is None else used_per_row
    assert used <= page_stride and R * used <= num_pages
    for L in lens:
        assert 0 <= L <= used * PAGE_SIZE
    gcpu = _gen(seed, "cpu")
    perm = torch.randperm(num_pages, generator=gcpu).to(torch.int32)
    pt = torch.full((R, page_stride), POISON_PAGE, dtype=torch.int32)
    for r in range(R):
        pt[r, :used] = perm[r * used:(r + 1) * used]
    ctx = torch.tensor(list(lens), dtype=torch.int32)
    T = R * B
    gdev = _gen(seed + 7919, device)
    qkv = _normal_bf16((T, (Hq + 2 * Hkv) * HEAD_DIM), gdev, device)
    pool = _normal_bf16((num_pages, 2, Hkv, PAGE_SIZE, HEAD_DIM), gdev, device)
    positions = qw = kw = None
    if qknorm:
        positions = torch.tensor([lens[r] + i for r in range(R) for i in range(B)], dtype=pos_dtype)
        qw = (1.0 + 0.1 * torch.randn(HEAD_DIM, generator=gcpu)).to(torch.bfloat16)
        kw = (1.0 + 0.1 * torch.randn(HEAD_DIM, generator=gcpu)).to(torch.bfloat16)
    case = Case(name=name, R=R, B=B, Hq=Hq, Hkv=Hkv, page_stride=page_stride,
                num_pages=num_pages, qknorm=qknorm, pos_dtype=pos_dtype, qkv=qkv, pool=pool,
                page_table=pt, ctx_lens=ctx, positions=positions, q_norm_w=qw, k_norm_w=kw)
    return case.to(device)


# ---- the workloads ---------------------------------------------------------

SPLITS = [(1, 8), (2, 4), (4, 2), (8, 1), (3, 5), (5, 3), (8, 8), (6, 6)]
SWEEP_LENGTHS = [0, 1, 63, 64, 65, 1000, 2041]


def tiny(device="cpu", seed: int = 0) -> Case:
    """1 request, block of 4, 6/1 heads, context 100 over 2 pages, q/k given
    already normalised and roped, softmax scale 1/8."""
    return build_case("tiny_1x4_6/1_L100", R=1, B=4, Hq=6, Hkv=1, lens=[100], page_stride=2,
                      num_pages=2, qknorm=False, seed=seed, device=device)


def mixed_8x8(device="cpu", seed: int = 1) -> Case:
    """8x8, 6/1, fused qknorm+RoPE, int32 positions, lengths U{0..2041},
    dense rows of a 4096-page pool."""
    g = _gen(seed + 101, "cpu")
    lens = torch.randint(0, 2042, (8,), generator=g).tolist()
    return build_case("mixed_8x8_6/1_L0-2041", R=8, B=8, Hq=6, Hkv=1, lens=lens, page_stride=32,
                      num_pages=4096, qknorm=True, pos_dtype=torch.int32, seed=seed, device=device)


def heads_24_4(device="cpu", seed: int = 2) -> Case:
    """8x8, 24/4, fused, int64 positions, every context 2041 tokens, strided
    rows (stride 40, 32 used, rest poisoned)."""
    return build_case("heads24/4_8x8_L2041_stride40", R=8, B=8, Hq=24, Hkv=4, lens=[2041] * 8,
                      page_stride=40, used_per_row=32, num_pages=4096, qknorm=True,
                      pos_dtype=torch.int64, seed=seed, device=device)


def split_sweep(R: int, B: int, device="cpu", seed: int = 3) -> Case:
    """One request x token split on 6/1 heads, lengths drawn per request from
    {0, 1, 63, 64, 65, 1000, 2041}, dense rows, fused, int32 positions."""
    g = _gen(seed + 211 * R + B, "cpu")
    idx = torch.randint(0, len(SWEEP_LENGTHS), (R,), generator=g).tolist()
    lens = [SWEEP_LENGTHS[k] for k in idx]
    return build_case(f"split_{R}x{B}_6/1", R=R, B=B, Hq=6, Hkv=1, lens=lens, page_stride=32,
                      num_pages=4096, qknorm=True, pos_dtype=torch.int32, seed=seed, device=device)


def long_context(device="cpu", seed: int = 4, num_pages: int = 20000, R: int = 8, B: int = 8,
                 lo: int = 16384, hi: int = 131072, page_stride: int = 2048) -> Case:
    """8x8, 24/4, fused, int64 positions, lengths U{16384..131072}, a
    20000-page pool, rows of a random page permutation (stride 2048)."""
    g = _gen(seed + 307, "cpu")
    lens = torch.randint(lo, hi + 1, (R,), generator=g).tolist()
    return build_case(f"long_{R}x{B}_24/4_L{lo // 1024}k-{hi // 1024}k_pool{num_pages}", R=R, B=B,
                      Hq=24, Hkv=4, lens=lens, page_stride=page_stride, num_pages=num_pages, qknorm=True,
                      pos_dtype=torch.int64, seed=seed, device=device)


def long_context_small(device="cpu", seed: int = 4) -> Case:
    """The long-context shape at a size meant for profiler captures: lengths
    U{16384..24576} (~160 MB of K/V read, more than L2), a 4096-page pool."""
    return long_context(device=device, seed=seed, num_pages=4096, lo=16384, hi=24576, page_stride=384)


def w6_8x6(device="cpu", seed: int = 5) -> Case:
    """The production draft block width W = 6: 8 requests x 6 tokens, 6/1
    heads (36 query rows per kv head), fused, int32 positions, lengths
    U{0..2041}, dense rows of a 4096-page pool."""
    g = _gen(seed + 401, "cpu")
    lens = torch.randint(0, 2042, (8,), generator=g).tolist()
    return build_case("w6_8x6_6/1_L0-2041", R=8, B=6, Hq=6, Hkv=1, lens=lens, page_stride=32,
                      num_pages=4096, qknorm=True, pos_dtype=torch.int32, seed=seed, device=device)


def single_w6(device="cpu", seed: int = 6, L: int = 2041, Hq: int = 6, Hkv: int = 1,
              page_stride: int = 32, num_pages: int = 4096) -> Case:
    """One request with a W = 6 block (the single-request case), fused,
    int64 positions; 6/1 heads and a 2041-token context by default."""
    return build_case(f"single_1x6_{Hq}/{Hkv}_L{L}", R=1, B=6, Hq=Hq, Hkv=Hkv, lens=[L],
                      page_stride=page_stride, num_pages=num_pages, qknorm=True,
                      pos_dtype=torch.int64, seed=seed, device=device)


def single_w6_long(device="cpu", seed: int = 7) -> Case:
    """One request, W = 6 block, 24/4 heads, a 32768-token context (512
    pages of a 4096-page pool)."""
    return single_w6(device=device, seed=seed, L=32768, Hq=24, Hkv=4, page_stride=512, num_pages=4096)


WORKLOADS = {
    "tiny": tiny,
    "mixed_8x8": mixed_8x8,
    "heads_24_4": heads_24_4,
    "long_context": long_context,
    "long_context_small": long_context_small,
    "w6_8x6": w6_8x6,
    "single_w6": single_w6,
    "single_w6_long": single_w6_long,
}

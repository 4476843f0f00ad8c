"""One call of the drafter block attention split into its independent
(request, kv head) units, each run through the fp64 oracle, on a pool of host
threads.

TEST INFRASTRUCTURE ONLY, like the rest of this package: the tests and the
CPU legs of ``bench.py`` call it; the product path never does.

Every unit is independent (page "[None][feat] Share Kimi K3 FP4 modeling and
add NVFP4 support on SM103", NVIDIA/TensorRT-LLM PR #20532, commit adding
k3_drafter_attn: each block token attends to its own request's context and
block only, and GQA maps query head h to kv head h / G), so the whole call's
output is the units' outputs laid side by side.  This module only selects
inputs (the unit's q, k and v heads, the request's pages and that kv head
of them) and places outputs; it does none of the method's arithmetic.  A CPU
test checks that the units reassemble the whole-request oracle output
exactly.

``case`` is any object with the attributes of a workload case: R, B, Hq, Hkv,
D, P, qknorm, scale, eps, rope_base, qkv, pool, page_table, ctx_lens,
positions, q_norm_w, k_norm_w (torch tensors, on any device).
"""
from __future__ import annotations

import os
import time
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from . import attn, bf16_bits, build


def _lens(case):
    return [int(x) for x in case.ctx_lens.cpu().tolist()]


def compact_unit(case, r: int, h: int) -> dict:
    """Request r, kv head h alone, as numpy arrays: its G query heads, its k
    and v heads of qkv, and kv head h of the pages its context occupies
    (renumbered 0..n-1 in context order)."""
    G, D, P, B = case.Hq // case.Hkv, case.D, case.P, case.B
    L = _lens(case)[r]
    n = (L + P - 1) // P
    rows = slice(r * B, (r + 1) * B)
    heads = list(range(h * G, (h + 1) * G)) + [case.Hq + h, case.Hq + case.Hkv + h]
    qkv = case.qkv[rows].reshape(B, case.Hq + 2 * case.Hkv, D)[:, heads].reshape(B, (G + 2) * D)
    if n:
        pages = case.page_table[r, :n].long().to(case.pool.device)
        pool = case.pool[pages, :, h:h + 1]
    else:
        pool = case.pool[:1, :, h:h + 1]
    pt = np.full((1, max(n, 1)), -1, dtype=np.int32)
    pt[0, :n] = np.arange(n, dtype=np.int32)
    unit = {"r": r, "h": h, "G": G, "B": B, "D": D, "qknorm": bool(case.qknorm), "scale": float(case.scale),
            "qkv": bf16_bits(qkv), "pool": bf16_bits(pool.contiguous()), "page_table": pt,
            "ctx_lens": np.array([L], dtype=np.int32), "tokens": L + B}
    if case.qknorm:
        unit.update(positions=case.positions[rows].cpu().numpy().astype(np.int64),
                    q_norm_w=bf16_bits(case.q_norm_w), k_norm_w=bf16_bits(case.k_norm_w),
                    eps=float(case.eps), rope_base=float(case.rope_base))
    return unit


def oracle_unit(u: dict) -> np.ndarray:
    """The oracle on one unit: ``[B, G*D]`` float64."""
    return attn(u["qkv"], u["pool"], u["page_table"], u["ctx_lens"], num_requests=1, block_len=u["B"],
                num_q_heads=u["G"], num_kv_heads=1, head_dim=u["D"], scale=u["scale"], qknorm=u["qknorm"],
                positions=u.get("positions"), q_norm_w=u.get("q_norm_w"), k_norm_w=u.get("k_norm_w"),
                eps=u.get("eps", 1e-5), rope_base=u.get("rope_base", 10000.0))


def units_of(case, requests=None):
    """The call's units (optionally of some requests only), longest first."""
    rs = range(case.R) if requests is None else requests
    return sorted((compact_unit(case, r, h) for r in rs for h in range(case.Hkv)), key=lambda u: -u["tokens"])


def host_threads() -> int:
    return len(os.sched_getaffinity(0))


def run_units(units, threads: int = 0):
    """Runs ``oracle_unit`` over ``units`` on ``threads`` host threads (all
    cores by default; the C oracle keeps no global state and ctypes releases
    the GIL during each call).  Returns (outputs in the order of ``units``,
    wall-clock seconds of the pool, threads used)."""
    build()
    n = threads or host_threads()
    with ThreadPoolExecutor(max_workers=n) as ex:
        list(ex.map(lambda _: None, range(n)))  # threads started before the clock
        t0 = time.perf_counter()
        outs = list(ex.map(oracle_unit, units))
        wall = time.perf_counter() - t0
    return outs, wall, n


def assemble(case, units, outs) -> np.ndarray:
    """Places unit outputs into the call's ``[T, Hq*D]`` layout (rows of
    requests without units stay NaN)."""
    G, D, B = case.Hq // case.Hkv, case.D, case.B
    out = np.full((case.R * B, case.Hq * D), np.nan)
    for u, o in zip(units, outs):
        out[u["r"] * B:(u["r"] + 1) * B, u["h"] * G * D:(u["h"] + 1) * G * D] = o
    return out


def oracle_call(case, threads: int = 0, requests=None) -> np.ndarray:
    """The whole call (or the rows of ``requests``) through the oracle, unit
    by unit on host threads: ``[T, Hq*D]`` float64."""
    units = units_of(case, requests)
    outs, _, _ = run_units(units, threads)
    return assemble(case, units, outs)

"""Host-side marshalling of the benchmark's oracle legs (CPU only): the
all-cores timing splits one call into (request, kv head) units, and each
unit's oracle output must be exactly that request's and heads' slice of
the whole-request oracle output."""
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import oracle  # noqa: E402
from speculative_decoding_drafter_k3_gb300 import workloads  # noqa: E402


def _whole_request(case, r):
    sub = bench.compact_request(case, r)
    return oracle.attn(sub.qkv, sub.pool, sub.page_table, sub.ctx_lens, num_requests=1,
                       block_len=sub.B, num_q_heads=sub.Hq, num_kv_heads=sub.Hkv, scale=sub.scale,
                       qknorm=sub.qknorm, positions=sub.positions, q_norm_w=sub.q_norm_w,
                       k_norm_w=sub.k_norm_w, eps=sub.eps, rope_base=sub.rope_base)


def test_units_reassemble_the_whole_request_exactly():
    case = workloads.build_case("units", R=3, B=5, Hq=24, Hkv=4, lens=[130, 0, 64], page_stride=4,
                                num_pages=12, qknorm=True, pos_dtype=torch.int64, seed=5)
    G, D = case.Hq // case.Hkv, case.D
    for r in range(case.R):
        whole = _whole_request(case, r)
        for h in range(case.Hkv):
            got = bench._oracle_unit(bench.compact_unit(case, r, h))
            assert np.array_equal(got, whole[:, h * G * D:(h + 1) * G * D])


def test_all_cores_timing_reports_its_threads():
    case = workloads.tiny()
    line = bench.cpu_all_cores(case, threads=2)
    assert line["cores"] == 2 and line["kind"] == "oracle" and line["value"] > 0
    assert "1 (request, kv head) units" in line["sample"]

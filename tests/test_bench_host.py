"""Host-side marshalling of the oracle's unit split (CPU only): a call split
into its (request, kv head) units and run unit by unit on host threads must
give exactly the oracle's whole-call output, and the benchmark's CPU legs
report what they ran."""
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import oracle  # noqa: E402
from oracle import units as ou  # noqa: E402
from speculative_decoding_drafter_k3_gb300 import workloads  # noqa: E402
from common import oracle_for  # noqa: E402


def test_units_reassemble_the_whole_call_exactly():
    case = workloads.build_case("units", R=3, B=5, Hq=24, Hkv=4, lens=[130, 0, 64], page_stride=4,
                                num_pages=12, qknorm=True, pos_dtype=torch.int64, seed=5)
    whole = oracle_for(case)
    assert np.array_equal(ou.oracle_call(case, threads=3), whole)
    # Some requests only: their rows are exact, the others stay unset.
    part = ou.oracle_call(case, threads=2, requests=[2])
    assert np.array_equal(part[10:15], whole[10:15]) and np.isnan(part[:10]).all()


def test_units_of_the_plain_variant_and_6_1_heads():
    case = workloads.split_sweep(5, 3, seed=9)
    case.qknorm = False
    assert np.array_equal(ou.oracle_call(case, threads=2), oracle_for(case))


def test_cpu_legs_report_their_threads_and_sample():
    case = workloads.tiny()
    line = bench.cpu_all_cores(case, threads=2)
    assert line["cores"] == 2 and line["kind"] == "oracle" and line["value"] > 0
    assert "whole call" in line["sample"] and "1 (request, kv head) units" in line["sample"]
    one = bench.cpu_baseline(case)
    assert one["cores"] == 1 and "whole call" in one["sample"]

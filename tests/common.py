"""Helpers shared by the GPU tests: the oracle call for a workloads.Case and
the tolerance check (2e-2 absolute + 2e-2 relative on bf16 outputs)."""
import numpy as np
import torch

import oracle

ATOL = 2e-2
RTOL = 2e-2


def oracle_for(case):
    return oracle.attn(case.qkv, case.pool, case.page_table.cpu(), case.ctx_lens.cpu(),
                       num_requests=case.R, block_len=case.B, num_q_heads=case.Hq,
                       num_kv_heads=case.Hkv, scale=case.scale, qknorm=case.qknorm,
                       positions=None if case.positions is None else case.positions.cpu(),
                       q_norm_w=case.q_norm_w, k_norm_w=case.k_norm_w, eps=case.eps,
                       rope_base=case.rope_base)


def assert_close(gpu_out, ref, what=""):
    g = gpu_out.detach().float().cpu().double().numpy().reshape(ref.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    err = np.abs(g - ref)
    bad = err > ATOL + RTOL * np.abs(ref)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {bad.sum()} elements outside {ATOL} abs + {RTOL} rel; "
                             f"max |err| {err.max():.3e}; first at {idx.tolist()}")
    return float(err.max())

"""Writes oracle_small.json: the oracle's output on small, fully
deterministic inputs (an integer hash, identical on every platform).

A regression fixture, not an independent pin: it guards the oracle against
accidental change.  It calls nothing but the oracle.
Run: python tests/golden/make_oracle_golden.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))
import oracle  # noqa: E402


def hashed_bf16_bits(n, salt):
    """bf16 bit patterns of values in [-2, 2) on a 1/64 grid, from a
    multiplicative hash of the index (exact in bf16)."""
    i = np.arange(n, dtype=np.uint64)
    h = ((i + np.uint64(salt)) * np.uint64(2654435761)) % np.uint64(1 << 32)
    vals = (h >> np.uint64(24)).astype(np.float32) / 64.0 - 2.0
    return (vals.view(np.uint32) >> 16).astype(np.uint16)


def problem():
    R, B, Hq, Hkv, D, P = 2, 3, 6, 1, 64, 64
    lens = np.array([70, 5], np.int32)
    pt = np.array([[2, 0], [1, -1]], np.int32)
    qkv = hashed_bf16_bits(R * B * (Hq + 2 * Hkv) * D, 11)
    pool = hashed_bf16_bits(3 * 2 * Hkv * P * D, 23)
    pos = np.array([lens[r] + i for r in range(R) for i in range(B)], np.int64)
    w = (np.full(D, 1.0, np.float32) + np.arange(D, dtype=np.float32) / 128.0)
    wb = (w.view(np.uint32) >> 16).astype(np.uint16)
    return dict(qkv=qkv, pool=pool, pt=pt, lens=lens, pos=pos, w=wb, R=R, B=B, Hq=Hq, Hkv=Hkv)


def compute(p, qknorm):
    return oracle.attn(p["qkv"], p["pool"], p["pt"], p["lens"], num_requests=p["R"],
                       block_len=p["B"], num_q_heads=p["Hq"], num_kv_heads=p["Hkv"],
                       qknorm=qknorm, positions=p["pos"], q_norm_w=p["w"], k_norm_w=p["w"][::-1].copy())


if __name__ == "__main__":
    p = problem()
    data = {"about": __doc__.strip().splitlines()[0],
            "plain": compute(p, False).reshape(-1).tolist(),
            "qknorm": compute(p, True).reshape(-1).tolist()}
    with open(os.path.join(HERE, "oracle_small.json"), "w") as f:
        json.dump(data, f)

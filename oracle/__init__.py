"""fp64 CPU oracle of the K3 DFlash drafter block attention (ctypes binding).

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are the only callers; the product path never
imports this package and shares no code with it.

The arithmetic lives in ``k3da_oracle.c`` (plain C, fp64, loops), which
follows the page "[None][feat] Share Kimi K3 FP4 modeling and add NVFP4
support on SM103" (NVIDIA/TensorRT-LLM PR #20532), the commit that adds the
drafter block attention ops and the commit that adds their contracts and the
fused_qk_norm_rope drafter cell.  This module only marshals numpy arrays into
that library and compiles it with gcc when the shared object is missing or
older than its source.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "k3da_oracle.c")
_LIB = os.path.join(_HERE, "libk3da_oracle.so")
_lock = threading.Lock()
_lib = None

# Error codes returned by k3o_attn.
OK, BAD_SHAPE, BAD_LENGTH, BAD_PAGE, NO_MEMORY = range(5)


def build(force: bool = False) -> str:
    """Compile the oracle into ``libk3da_oracle.so`` beside its source."""
    stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        # -ffp-contract=off: no fused multiply-add contraction, so x86 and Arm
        # builds round every fp64 step the same way.
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            dp = ctypes.POINTER(ctypes.c_double)
            lib.k3o_rmsnorm.argtypes = [dp, dp, ctypes.c_int, ctypes.c_double, dp]
            lib.k3o_rmsnorm.restype = None
            lib.k3o_rope_neox.argtypes = [dp, ctypes.c_int, ctypes.c_double, ctypes.c_double, dp]
            lib.k3o_rope_neox.restype = None
            vp = ctypes.c_void_p
            lib.k3o_attn.argtypes = [
                vp, vp, vp, ctypes.c_int64, vp, ctypes.c_int, vp,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_double, ctypes.c_int, vp, vp, vp,
                ctypes.c_double, ctypes.c_double,
            ]
            lib.k3o_attn.restype = ctypes.c_int
            lib.k3o_qk_norm_rope.argtypes = [
                vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp, vp,
                ctypes.c_double, ctypes.c_double,
            ]
            lib.k3o_qk_norm_rope.restype = ctypes.c_int
            d = ctypes.c_double
            lib.k3o_yarn_inv_freq.argtypes = [dp, ctypes.c_int, d, d, d, d, d]
            lib.k3o_yarn_inv_freq.restype = None
            lib.k3o_rope_table.argtypes = [dp, ctypes.c_int, d, dp, d, dp]
            lib.k3o_rope_table.restype = None
            lib.k3o_attn_yarn.argtypes = [
                vp, vp, vp, ctypes.c_int64, vp, ctypes.c_int, vp,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, d, vp, vp, vp, d, d, d, d, d, d, d,
            ]
            lib.k3o_attn_yarn.restype = ctypes.c_int
            lib.k3o_qk_norm_rope_yarn.argtypes = [
                vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp, vp,
                d, d, d, d, d, d, d,
            ]
            lib.k3o_qk_norm_rope_yarn.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def rmsnorm(x, w, eps: float = 1e-5) -> np.ndarray:
    """RMSNorm of one head row (fp64): x * (mean(x^2) + eps)^-1/2 * w."""
    lib = _load()
    x = _f64(x)
    w = _f64(w)
    assert x.ndim == 1 and w.shape == x.shape
    y = np.empty_like(x)
    dp = ctypes.POINTER(ctypes.c_double)
    lib.k3o_rmsnorm(x.ctypes.data_as(dp), w.ctypes.data_as(dp), x.shape[0], float(eps),
                    y.ctypes.data_as(dp))
    return y


def rope_neox(x, pos: float, base: float = 10000.0) -> np.ndarray:
    """NeoX RoPE of one head row at position ``pos`` (fp64)."""
    lib = _load()
    x = _f64(x)
    assert x.ndim == 1 and x.shape[0] % 2 == 0
    y = np.empty_like(x)
    dp = ctypes.POINTER(ctypes.c_double)
    lib.k3o_rope_neox(x.ctypes.data_as(dp), x.shape[0], float(pos), float(base),
                      y.ctypes.data_as(dp))
    return y


def yarn_inv_freq(D: int, base: float, factor: float, original_max_position: float,
                  beta_fast: float = 32.0, beta_slow: float = 1.0) -> np.ndarray:
    """YaRN rotary frequencies of the D/2 pairs (fp64)."""
    lib = _load()
    inv = np.empty(D // 2, dtype=np.float64)
    dp = ctypes.POINTER(ctypes.c_double)
    lib.k3o_yarn_inv_freq(inv.ctypes.data_as(dp), D, float(base), float(factor),
                          float(original_max_position), float(beta_slow), float(beta_fast))
    return inv


def rope_table(x, pos: float, inv_freq, mscale: float = 1.0) -> np.ndarray:
    """Rotary embedding of one head row with an explicit frequency table,
    both outputs scaled by ``mscale`` (fp64)."""
    lib = _load()
    x = _f64(x)
    inv = _f64(inv_freq)
    assert x.ndim == 1 and inv.shape[0] == x.shape[0] // 2
    y = np.empty_like(x)
    dp = ctypes.POINTER(ctypes.c_double)
    lib.k3o_rope_table(x.ctypes.data_as(dp), x.shape[0], float(pos), inv.ctypes.data_as(dp),
                       float(mscale), y.ctypes.data_as(dp))
    return y


def bf16_bits(a) -> np.ndarray:
    """uint16 bit patterns of a bf16 torch tensor, or a uint16 array as is."""
    if isinstance(a, np.ndarray):
        assert a.dtype == np.uint16
        return np.ascontiguousarray(a)
    import torch  # only for the view; no arithmetic

    assert a.dtype == torch.bfloat16
    return np.ascontiguousarray(a.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def attn(qkv, pool, page_table, ctx_lens, *, num_requests: int, block_len: int,
         num_q_heads: int, num_kv_heads: int, head_dim: int = 64, page_size: int = 64,
         scale: float = 0.125, qknorm: bool = False, positions=None, q_norm_w=None,
         k_norm_w=None, eps: float = 1e-5, rope_base: float = 10000.0,
         check: bool = True, yarn=None):
    """Drafter block attention in fp64; returns ``[T, Hq*D]`` float64.

    ``qkv``, ``pool``, ``q_norm_w`` and ``k_norm_w`` are bf16 (torch tensors or
    uint16 bit arrays); ``page_table`` is ``[R, S]`` int32, ``ctx_lens`` ``[R]``
    int32, ``positions`` ``[T]`` of any integer type.  With ``check`` a nonzero
    status raises ``ValueError``; without it ``(out, status)`` is returned.
    """
    lib = _load()
    R, B, Hq, Hkv, D = num_requests, block_len, num_q_heads, num_kv_heads, head_dim
    T = R * B
    qkv_b = bf16_bits(qkv).reshape(-1)
    pool_b = bf16_bits(pool).reshape(-1)
    pt = np.ascontiguousarray(np.asarray(_np(page_table), dtype=np.int32))
    assert pt.ndim == 2 and pt.shape[0] == R
    lens = np.ascontiguousarray(np.asarray(_np(ctx_lens), dtype=np.int32).reshape(-1))
    assert lens.shape[0] == R
    assert qkv_b.shape[0] == T * (Hq + 2 * Hkv) * D
    per_page = 2 * Hkv * page_size * D
    assert pool_b.shape[0] % per_page == 0
    num_pages = pool_b.shape[0] // per_page
    if qknorm:
        pos = np.ascontiguousarray(np.asarray(_np(positions)).astype(np.int64).reshape(-1))
        assert pos.shape[0] == T
        qw = bf16_bits(q_norm_w).reshape(-1)
        kw = bf16_bits(k_norm_w).reshape(-1)
        assert qw.shape[0] == D and kw.shape[0] == D
        pos_p, qw_p, kw_p = _ptr(pos), _ptr(qw), _ptr(kw)
    else:
        pos_p = qw_p = kw_p = None
    out = np.zeros((T, Hq * D), dtype=np.float64)
    if yarn is not None:
        # ``yarn``: dict(factor, original_max_position, beta_fast, beta_slow, mscale).
        assert qknorm, "YaRN applies to the fused variant"
        st = lib.k3o_attn_yarn(_ptr(out), _ptr(qkv_b), _ptr(pool_b), num_pages, _ptr(pt), pt.shape[1],
                               _ptr(lens), R, B, Hq, Hkv, D, page_size, float(scale), pos_p, qw_p, kw_p,
                               float(eps), float(rope_base), float(yarn["factor"]),
                               float(yarn["original_max_position"]), float(yarn["beta_fast"]),
                               float(yarn["beta_slow"]), float(yarn["mscale"]))
    else:
        st = lib.k3o_attn(_ptr(out), _ptr(qkv_b), _ptr(pool_b), num_pages, _ptr(pt), pt.shape[1],
                          _ptr(lens), R, B, Hq, Hkv, D, page_size, float(scale), int(bool(qknorm)),
                          pos_p, qw_p, kw_p, float(eps), float(rope_base))
    if check:
        if st != OK:
            raise ValueError(f"oracle refused the inputs (status {st})")
        return out
    return out, st


def qk_norm_rope(qkv, positions, q_norm_w, k_norm_w, *, num_q_heads: int, num_kv_heads: int,
                 head_dim: int = 64, eps: float = 1e-5, rope_base: float = 10000.0,
                 yarn=None) -> np.ndarray:
    """The fused q/k norm + RoPE cell in fp64: ``[T, (Hq+2Hkv)*D]`` float64
    with q and k heads normalised and rotated at their token's position and
    v heads copied.  ``qkv``, ``q_norm_w``, ``k_norm_w`` are bf16; positions
    of any integer type."""
    lib = _load()
    Hq, Hkv, D = num_q_heads, num_kv_heads, head_dim
    qkv_b = bf16_bits(qkv).reshape(-1)
    W = (Hq + 2 * Hkv) * D
    assert qkv_b.shape[0] % W == 0
    T = qkv_b.shape[0] // W
    pos = np.ascontiguousarray(np.asarray(_np(positions)).astype(np.int64).reshape(-1))
    assert pos.shape[0] == T
    qw = bf16_bits(q_norm_w).reshape(-1)
    kw = bf16_bits(k_norm_w).reshape(-1)
    assert qw.shape[0] == D and kw.shape[0] == D
    out = np.zeros((T, W), dtype=np.float64)
    if yarn is not None:
        st = lib.k3o_qk_norm_rope_yarn(_ptr(out), _ptr(qkv_b), T, Hq, Hkv, D, _ptr(pos), _ptr(qw), _ptr(kw),
                                       float(eps), float(rope_base), float(yarn["factor"]),
                                       float(yarn["original_max_position"]), float(yarn["beta_fast"]),
                                       float(yarn["beta_slow"]), float(yarn["mscale"]))
    else:
        st = lib.k3o_qk_norm_rope(_ptr(out), _ptr(qkv_b), T, Hq, Hkv, D, _ptr(pos), _ptr(qw), _ptr(kw),
                                  float(eps), float(rope_base))
    if st != OK:
        raise ValueError(f"oracle refused the inputs (status {st})")
    return out


def _np(a):
    """numpy view of a CPU torch tensor or array-like (no arithmetic)."""
    if hasattr(a, "detach"):
        return a.detach().cpu().numpy()
    return a

"""K3 DFlash drafter block attention on sm_103a: thin Python binding.

The compute lives in ``libk3da.so`` (hand-written CUDA, C ABI declared in
``include/k3da.h``).  This module only marshals torch tensors into that ABI:
pointers (device memory, or pinned host memory where the ABI allows it),
sizes, dtype codes and the current CUDA stream.  There is no
CPU fallback: if the library is missing, every call raises.

Operation (page "[None][feat] Share Kimi K3 FP4 modeling and add NVFP4
support on SM103", NVIDIA/TensorRT-LLM PR #20532, commit adding
k3_drafter_attn / k3_drafter_attn_qknorm): each of R <= 8 requests brings a
block of B <= 8 draft tokens; every block token attends densely to its
request's paged context (HND pages of 64) and to its own block's K/V, taken
from qkv and never written to the pool; GQA 6:1 (6/1 or 24/4 heads),
head_dim 64.  ``k3da_attn_qknorm`` first applies per-head q/k RMSNorm and
NeoX RoPE.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = [
    "K3daError", "library_path", "load_library", "workspace_bytes", "k3da_attn",
    "k3da_attn_qknorm", "STATUS_BAD_LENGTH", "STATUS_BAD_PAGE", "STATUS_TIMEOUT",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libk3da.so")
_lock = threading.Lock()
_lib = None

OK, EINVAL, EUNSUPPORTED, ECUDA, EWORKSPACE = 0, -1, -2, -3, -4
STATUS_BAD_LENGTH, STATUS_BAD_PAGE, STATUS_TIMEOUT = 1, 2, 4
POS_I32, POS_I64 = 0, 1
EXPORTED = ["k3da_workspace_bytes", "k3da_attn", "k3da_attn_qknorm", "k3da_attn_qknorm_noalloc",
            "k3da_noalloc_scratch_bytes", "k3da_split_grid", "k3da_set_phase_event",
            "k3da_error_string", "k3da_version", "k3da_qk_norm_rope", "k3da_attn_qknorm_yarn",
            "k3da_qk_norm_rope_yarn", "k3da_selftest_wait_timeout"]


class Yarn(ctypes.Structure):
    """k3da_yarn: YaRN RoPE scaling (factor, original_max_position, beta_fast,
    beta_slow, mscale).  mscale 0 asks the library for the YaRN paper's
    default multiplier."""
    _fields_ = [("factor", ctypes.c_float), ("original_max_position", ctypes.c_float),
                ("beta_fast", ctypes.c_float), ("beta_slow", ctypes.c_float), ("mscale", ctypes.c_float)]

    @classmethod
    def of(cls, factor: float, original_max_position: float, beta_fast: float = 32.0,
           beta_slow: float = 1.0, mscale: float = 0.0):
        return cls(factor, original_max_position, beta_fast, beta_slow, mscale)

    def as_dict(self):
        return {k: float(getattr(self, k)) for k, _ in self._fields_}


class K3daError(ValueError):
    """A call refused by the library (host-side check) or a device status."""


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load libk3da.so (ctypes) and declare its signatures; raise if absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"{_LIB_PATH} is missing: build it with "
                "`python -m speculative_decoding_drafter_k3_gb300.build` (there is no CPU fallback)")
        lib = ctypes.CDLL(_LIB_PATH)
        c_int, c_i64, c_sz, vp, c_f = (ctypes.c_int, ctypes.c_int64, ctypes.c_size_t,
                                       ctypes.c_void_p, ctypes.c_float)
        lib.k3da_workspace_bytes.argtypes = [c_int, c_int, c_int, c_int, c_int]
        lib.k3da_workspace_bytes.restype = c_sz
        common = [vp, vp, vp, c_i64, vp, c_int, vp, c_int, c_int, c_int, c_int, c_int, c_f]
        lib.k3da_attn.argtypes = common + [vp, c_sz, vp, vp]
        lib.k3da_attn.restype = c_int
        lib.k3da_attn_qknorm.argtypes = common + [vp, c_int, vp, vp, c_f, c_f, vp, c_sz, vp, vp]
        lib.k3da_attn_qknorm.restype = c_int
        lib.k3da_error_string.argtypes = [c_int]
        lib.k3da_error_string.restype = ctypes.c_char_p
        lib.k3da_attn_qknorm_noalloc.argtypes = common + [vp, c_int, vp, vp, c_f, c_f, vp, vp]
        lib.k3da_attn_qknorm_noalloc.restype = c_int
        lib.k3da_noalloc_scratch_bytes.argtypes = []
        lib.k3da_noalloc_scratch_bytes.restype = c_sz
        lib.k3da_split_grid.argtypes = [c_int]
        lib.k3da_split_grid.restype = c_int
        lib.k3da_set_phase_event.argtypes = [vp]
        lib.k3da_set_phase_event.restype = c_int
        lib.k3da_version.argtypes = []
        lib.k3da_version.restype = c_int
        lib.k3da_qk_norm_rope.argtypes = [vp, c_int, c_int, c_int, c_int, vp, c_int, vp, vp, c_f, c_f, vp]
        lib.k3da_qk_norm_rope.restype = c_int
        yp = ctypes.POINTER(Yarn)
        lib.k3da_attn_qknorm_yarn.argtypes = common + [vp, c_int, vp, vp, c_f, c_f, yp, vp, c_sz, vp, vp]
        lib.k3da_attn_qknorm_yarn.restype = c_int
        lib.k3da_qk_norm_rope_yarn.argtypes = [vp, c_int, c_int, c_int, c_int, vp, c_int, vp, vp, c_f, c_f, yp, vp]
        lib.k3da_qk_norm_rope_yarn.restype = c_int
        lib.k3da_selftest_wait_timeout.argtypes = [vp, ctypes.c_ulonglong, vp]
        lib.k3da_selftest_wait_timeout.restype = c_int
        _lib = lib
        return lib


def error_string(code: int) -> str:
    return load_library().k3da_error_string(int(code)).decode()


def _check(rc: int, what: str):
    if rc != OK:
        raise K3daError(f"{what}: {error_string(rc)} (code {rc})")


def workspace_bytes(num_requests: int, block_len: int, num_q_heads: int, num_kv_heads: int,
                    page_stride: int) -> int:
    n = load_library().k3da_workspace_bytes(num_requests, block_len, num_q_heads, num_kv_heads,
                                            page_stride)
    if n == 0:
        raise K3daError("workspace_bytes: sizes out of contract")
    return int(n)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _device_or_pinned(name, t):
    """out, qkv, page_table, ctx_lens and positions may live in pinned host
    memory, which the kernels read (or write) across the host link."""
    if not (t.is_cuda or t.is_pinned()) or not t.is_contiguous():
        raise K3daError(f"{name} must be a contiguous CUDA tensor or a contiguous pinned host tensor")


def _device_scratch(workspace, status):
    """The workspace and the status word are always device memory."""
    if workspace is not None and (not workspace.is_cuda or not workspace.is_contiguous()):
        raise K3daError("workspace must be a contiguous CUDA tensor")
    if status is not None and (not status.is_cuda or status.dtype != torch.int32):
        raise K3daError("status must be an int32 CUDA tensor")


def _shape_args(out, qkv, kv_pool, page_table, ctx_lens, block_len, num_q_heads, num_kv_heads):
    for name, t in [("out", out), ("qkv", qkv), ("page_table", page_table), ("ctx_lens", ctx_lens)]:
        _device_or_pinned(name, t)
    if not kv_pool.is_cuda or not kv_pool.is_contiguous():
        raise K3daError("kv_pool must be a contiguous CUDA tensor")
    if qkv.dtype != torch.bfloat16 or out.dtype != torch.bfloat16 or kv_pool.dtype != torch.bfloat16:
        raise K3daError("qkv, out and kv_pool must be bf16")
    if page_table.dtype != torch.int32 or ctx_lens.dtype != torch.int32:
        raise K3daError("page_table and ctx_lens must be int32")
    if page_table.dim() != 2 or kv_pool.dim() != 5:
        raise K3daError("page_table must be [R, S] and kv_pool [pages, 2, Hkv, 64, 64]")
    R = page_table.shape[0]
    T = R * block_len
    D = kv_pool.shape[-1]
    if (tuple(kv_pool.shape[1:]) != (2, num_kv_heads, 64, D) or ctx_lens.numel() != R
            or tuple(qkv.shape) != (T, (num_q_heads + 2 * num_kv_heads) * D)
            or tuple(out.shape) != (T, num_q_heads * D)):
        raise K3daError("tensor shapes disagree with (R, B, Hq, Hkv, head_dim)")
    return R, kv_pool.shape[0], page_table.shape[1], D


def _qknorm_args(positions, q_norm_w, k_norm_w, T, D):
    """Checks the fused variant's extra tensors; returns the positions' dtype code."""
    if positions.dtype not in (torch.int32, torch.int64) or positions.numel() != T:
        raise K3daError("positions must be [T] int32 or int64")
    _device_or_pinned("positions", positions)
    for name, t in [("q_norm_w", q_norm_w), ("k_norm_w", k_norm_w)]:
        if not t.is_cuda or not t.is_contiguous():
            raise K3daError(f"{name} must be a contiguous CUDA tensor")
    if q_norm_w.dtype != torch.bfloat16 or k_norm_w.dtype != torch.bfloat16 or \
            q_norm_w.numel() != D or k_norm_w.numel() != D:
        raise K3daError("norm weights must be [64] bf16")
    return POS_I64 if positions.dtype == torch.int64 else POS_I32


def k3da_attn(out, qkv, kv_pool, page_table, ctx_lens, *, block_len: int, num_q_heads: int,
              num_kv_heads: int, softmax_scale: float = 0.125, workspace, status=None,
              stream=None):
    """Block attention on already normalised and roped q/k (C: k3da_attn)."""
    lib = load_library()
    R, num_pages, S, D = _shape_args(out, qkv, kv_pool, page_table, ctx_lens, block_len,
                                     num_q_heads, num_kv_heads)
    _device_scratch(workspace, status)
    rc = lib.k3da_attn(_ptr(out), _ptr(qkv), _ptr(kv_pool), num_pages, _ptr(page_table), S,
                       _ptr(ctx_lens), R, block_len, num_q_heads, num_kv_heads, D,
                       float(softmax_scale), _ptr(workspace), workspace.numel() * workspace.element_size(),
                       _ptr(status), _stream(stream))
    _check(rc, "k3da_attn")
    return out


def k3da_attn_qknorm(out, qkv, kv_pool, page_table, ctx_lens, positions, q_norm_w, k_norm_w, *,
                     block_len: int, num_q_heads: int, num_kv_heads: int,
                     softmax_scale: float = 0.125, eps: float = 1e-5, rope_base: float = 10000.0,
                     workspace, status=None, stream=None, yarn=None):
    """Block attention with fused q/k RMSNorm + NeoX RoPE (C: k3da_attn_qknorm);
    with ``yarn`` (a ``Yarn``), YaRN RoPE (C: k3da_attn_qknorm_yarn)."""
    lib = load_library()
    R, num_pages, S, D = _shape_args(out, qkv, kv_pool, page_table, ctx_lens, block_len,
                                     num_q_heads, num_kv_heads)
    _device_scratch(workspace, status)
    pos_code = _qknorm_args(positions, q_norm_w, k_norm_w, R * block_len, D)
    args = [_ptr(out), _ptr(qkv), _ptr(kv_pool), num_pages, _ptr(page_table), S, _ptr(ctx_lens), R,
            block_len, num_q_heads, num_kv_heads, D, float(softmax_scale), _ptr(positions), pos_code,
            _ptr(q_norm_w), _ptr(k_norm_w), float(eps), float(rope_base)]
    tail = [_ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(status), _stream(stream)]
    if yarn is None:
        rc = lib.k3da_attn_qknorm(*args, *tail)
        _check(rc, "k3da_attn_qknorm")
    else:
        rc = lib.k3da_attn_qknorm_yarn(*args, ctypes.byref(yarn), *tail)
        _check(rc, "k3da_attn_qknorm_yarn")
    return out


def k3da_qk_norm_rope(qkv, positions, q_norm_w, k_norm_w, *, num_q_heads: int, num_kv_heads: int,
                      eps: float = 1e-5, rope_base: float = 10000.0, stream=None, yarn=None):
    """The fused q/k RMSNorm + NeoX RoPE cell, in place on the q and k heads
    of ``qkv`` ``[T, (Hq+2Hkv)*64]`` bf16 (C: k3da_qk_norm_rope); with
    ``yarn`` (a ``Yarn``), YaRN RoPE (C: k3da_qk_norm_rope_yarn)."""
    lib = load_library()
    for name, t in [("qkv", qkv), ("positions", positions), ("q_norm_w", q_norm_w), ("k_norm_w", k_norm_w)]:
        if not t.is_cuda or not t.is_contiguous():
            raise K3daError(f"{name} must be a contiguous CUDA tensor")
    if qkv.dtype != torch.bfloat16 or qkv.dim() != 2:
        raise K3daError("qkv must be [T, (Hq+2Hkv)*64] bf16")
    D = qkv.shape[1] // (num_q_heads + 2 * num_kv_heads)
    T = qkv.shape[0]
    if positions.dtype not in (torch.int32, torch.int64) or positions.numel() != T:
        raise K3daError("positions must be [T] int32 or int64")
    if q_norm_w.dtype != torch.bfloat16 or k_norm_w.dtype != torch.bfloat16 or \
            q_norm_w.numel() != D or k_norm_w.numel() != D:
        raise K3daError("norm weights must be [head_dim] bf16")
    pos_code = POS_I64 if positions.dtype == torch.int64 else POS_I32
    args = [_ptr(qkv), T, num_q_heads, num_kv_heads, D, _ptr(positions), pos_code, _ptr(q_norm_w),
            _ptr(k_norm_w), float(eps), float(rope_base)]
    if yarn is None:
        rc = lib.k3da_qk_norm_rope(*args, _stream(stream))
        _check(rc, "k3da_qk_norm_rope")
    else:
        rc = lib.k3da_qk_norm_rope_yarn(*args, ctypes.byref(yarn), _stream(stream))
        _check(rc, "k3da_qk_norm_rope_yarn")
    return qkv


def alloc_workspace(num_requests: int, block_len: int, num_q_heads: int, num_kv_heads: int,
                    page_stride: int, device=None) -> torch.Tensor:
    """A workspace tensor (uint8, 256-byte aligned by torch) for these sizes."""
    device = torch.device("cuda") if device is None else torch.device(device)
    n = workspace_bytes(num_requests, block_len, num_q_heads, num_kv_heads, page_stride)
    return torch.empty(n, dtype=torch.uint8, device=device)


def case_workspace(case) -> torch.Tensor:
    return alloc_workspace(case.R, case.B, case.Hq, case.Hkv, case.page_stride, case.pool.device)


def run_case(case, out=None, workspace=None, status=None, stream=None, yarn=None):
    """Run the op on a ``workloads.Case`` whose pool and norm weights are on
    the GPU; its qkv, page table, lengths and positions may be pinned host
    tensors (``yarn``: YaRN RoPE for the fused variant)."""
    if out is None:
        out = torch.empty(case.T, case.Hq * case.D, dtype=torch.bfloat16, device=case.pool.device)
    if workspace is None:
        workspace = case_workspace(case)
    kw = dict(block_len=case.B, num_q_heads=case.Hq, num_kv_heads=case.Hkv,
              softmax_scale=case.scale, workspace=workspace, status=status, stream=stream)
    if case.qknorm:
        return k3da_attn_qknorm(out, case.qkv, case.pool, case.page_table, case.ctx_lens,
                                case.positions, case.q_norm_w, case.k_norm_w, eps=case.eps,
                                rope_base=case.rope_base, yarn=yarn, **kw)
    return k3da_attn(out, case.qkv, case.pool, case.page_table, case.ctx_lens, **kw)


def set_phase_event(event):
    """Record ``event`` (a torch.cuda.Event) between the split pass and the
    combine of every later call from this thread; None turns it off."""
    if event is None:
        handle = None
    else:
        handle = ctypes.c_void_p(event.cuda_event)
    _check(load_library().k3da_set_phase_event(handle), "k3da_set_phase_event")


def split_grid(device: int = -1) -> int:
    """CTAs the split pass launches on ``device`` (SMs x CTAs per SM)."""
    return int(load_library().k3da_split_grid(device))


def k3da_attn_qknorm_noalloc(out, qkv, kv_pool, page_table, ctx_lens, positions, q_norm_w, k_norm_w, *,
                             block_len: int, num_q_heads: int, num_kv_heads: int,
                             softmax_scale: float = 0.125, eps: float = 1e-5,
                             rope_base: float = 10000.0, status=None, stream=None):
    """k3da_attn_qknorm without a workspace argument, for callers that cannot
    allocate: the library's fixed per-GPU scratch array is used instead
    (C: k3da_attn_qknorm_noalloc; calls that overlap on the GPU race on it)."""
    lib = load_library()
    R, num_pages, S, D = _shape_args(out, qkv, kv_pool, page_table, ctx_lens, block_len,
                                     num_q_heads, num_kv_heads)
    _device_scratch(None, status)
    pos_code = _qknorm_args(positions, q_norm_w, k_norm_w, R * block_len, D)
    rc = lib.k3da_attn_qknorm_noalloc(_ptr(out), _ptr(qkv), _ptr(kv_pool), num_pages, _ptr(page_table),
                                      S, _ptr(ctx_lens), R, block_len, num_q_heads, num_kv_heads, D,
                                      float(softmax_scale), _ptr(positions), pos_code, _ptr(q_norm_w),
                                      _ptr(k_norm_w), float(eps), float(rope_base), _ptr(status),
                                      _stream(stream))
    _check(rc, "k3da_attn_qknorm_noalloc")
    return out

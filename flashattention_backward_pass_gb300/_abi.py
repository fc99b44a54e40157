"""ctypes binding of the C ABI in include/fa.h (argument marshalling only).

Every step of the forward and backward runs in the CUDA kernels of libfa_gb300.so;
this module only turns torch tensors into `fa_tensor` views, allocates the caller-side
workspace with torch, and passes the current CUDA stream.  It raises when the library
is missing: there is no fallback implementation.
"""

from __future__ import annotations

import ctypes
import os
import re

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfa_gb300.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "fa.h")

FA_DTYPE_BF16 = 0
FA_DTYPE_FP32 = 1
FA_DTYPE_F16 = 2

STATUS = {
    0: "FA_OK", -1: "FA_ERR_NULL", -2: "FA_ERR_SHAPE", -3: "FA_ERR_DTYPE", -4: "FA_ERR_HEADDIM",
    -5: "FA_ERR_LAYOUT", -6: "FA_ERR_ALIGNMENT", -7: "FA_ERR_WORKSPACE", -8: "FA_ERR_UNSUPPORTED",
    -9: "FA_ERR_ARG", -10: "FA_ERR_CUDA", -11: "FA_ERR_DEVICE_TIMEOUT",
}


class FaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} ({status})")


class FaTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("shape", ctypes.c_int64 * 4),
                ("stride", ctypes.c_int64 * 4), ("ndim", ctypes.c_int32),
                ("dtype", ctypes.c_int32)]


_lib = None


def load(path: str = LIB_PATH):
    """Load libfa_gb300.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER(FaTensor)
    vp, sz = ctypes.c_void_p, ctypes.c_size_t
    lib.fa_abi_version.restype = ctypes.c_int
    lib.fa_status_string.restype = ctypes.c_char_p
    lib.fa_status_string.argtypes = [ctypes.c_int]
    lib.fa_fwd_workspace_size.restype = sz
    lib.fa_fwd_workspace_size.argtypes = [ctypes.c_int] * 6
    lib.fa_bwd_workspace_size.restype = sz
    lib.fa_bwd_workspace_size.argtypes = [ctypes.c_int] * 7
    lib.fa_bwd_workspace_size_dv.restype = sz
    lib.fa_bwd_workspace_size_dv.argtypes = [ctypes.c_int] * 8
    lib.fa_fwd.restype = ctypes.c_int
    lib.fa_fwd.argtypes = [P, P, P, P, P, ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                           ctypes.c_float, vp, sz, vp]
    lib.fa_bwd.restype = ctypes.c_int
    lib.fa_bwd.argtypes = [P, P, P, P, P, P, P, P, P, ctypes.c_float, ctypes.c_int, ctypes.c_int,
                           ctypes.c_int, ctypes.c_float, ctypes.c_int, vp, sz, vp]
    lib.fa_bwd_status.restype = ctypes.c_int
    lib.fa_bwd_status.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_int)]
    lib.fa_debug_set_wait_limit.restype = ctypes.c_int
    lib.fa_debug_set_wait_limit.argtypes = [ctypes.c_longlong]
    lib.fa_debug_poison_ordering.restype = ctypes.c_int
    lib.fa_debug_poison_ordering.argtypes = [ctypes.c_int]
    lib.fa_profile_enable.restype = ctypes.c_int
    lib.fa_profile_enable.argtypes = [ctypes.c_int]
    lib.fa_profile_read.restype = ctypes.c_int
    lib.fa_profile_read.argtypes = [ctypes.POINTER(ctypes.c_float)]
    lib.fa_bwd_set_algorithm.restype = ctypes.c_int
    lib.fa_bwd_set_algorithm.argtypes = [ctypes.c_int]
    lib.fa_bwd_get_algorithm.restype = ctypes.c_int
    ip = ctypes.c_void_p  # device int32 offsets
    lib.fa_fwd_varlen.restype = ctypes.c_int
    lib.fa_fwd_varlen.argtypes = [P, P, P, P, P, ip, ip, ip, ip, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                  ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                  ctypes.c_float, vp, sz, vp]
    lib.fa_bwd_varlen_workspace_size.restype = sz
    lib.fa_bwd_varlen_workspace_size.argtypes = [ctypes.c_int] * 5
    lib.fa_fwd_blocksparse.restype = ctypes.c_int
    lib.fa_fwd_blocksparse.argtypes = [P, P, P, P, P, vp, ctypes.c_float, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int, ctypes.c_float, vp, sz, vp]
    lib.fa_bwd_blocksparse_workspace_size.restype = sz
    lib.fa_bwd_blocksparse_workspace_size.argtypes = [ctypes.c_int] * 6
    lib.fa_bwd_blocksparse.restype = ctypes.c_int
    lib.fa_bwd_blocksparse.argtypes = [P, P, P, P, P, P, P, P, P, vp, ctypes.c_float, ctypes.c_int,
                                       ctypes.c_int, ctypes.c_int, ctypes.c_float, ctypes.c_int,
                                       vp, sz, vp]
    lib.fa_bwd_varlen.restype = ctypes.c_int
    lib.fa_bwd_varlen.argtypes = [P, P, P, P, P, P, P, P, P, ip, ip, ip, ip, ctypes.c_int, ctypes.c_int,
                                  ctypes.c_int, ctypes.c_float, ctypes.c_int, ctypes.c_int,
                                  ctypes.c_int, ctypes.c_float, ctypes.c_int, vp, sz, vp]
    lib.fa_bwd_noalloc.restype = ctypes.c_int
    lib.fa_bwd_noalloc.argtypes = [P, P, P, P, P, P, P, P, P, ctypes.c_float, ctypes.c_int,
                                   ctypes.c_int, ctypes.c_int, ctypes.c_float, ctypes.c_int, vp]
    lib.fa_bwd_noalloc_status.restype = ctypes.c_int
    lib.fa_bwd_noalloc_status.argtypes = [vp, ctypes.POINTER(ctypes.c_int)]
    if lib.fa_abi_version() != 3:
        raise RuntimeError(f"{path} reports ABI version {lib.fa_abi_version()}, expected 3: rebuild it")
    _lib = lib
    return lib


def declared_functions(header: str = HEADER_PATH):
    """Names of the functions include/fa.h declares."""
    with open(header) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(fa_[a-z0-9_]+)\s*\(",
                                 text, flags=re.M)))


def tensor_view(t: torch.Tensor) -> FaTensor:
    if t.dtype == torch.bfloat16:
        dt = FA_DTYPE_BF16
    elif t.dtype == torch.float32:
        dt = FA_DTYPE_FP32
    elif t.dtype == torch.float16:
        dt = FA_DTYPE_F16
    else:
        dt = 99
    v = FaTensor()
    v.data = t.data_ptr() if t.numel() > 0 else None
    for i in range(4):
        v.shape[i] = t.shape[i] if i < t.dim() else 0
        v.stride[i] = t.stride(i) if i < t.dim() else 0
    v.ndim = t.dim()
    v.dtype = dt
    return v


def _stream_ptr(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(st: int, where: str):
    if st != 0:
        raise FaError(st, where)


def bwd_workspace_size(B, H, Hk, Sq, Sk, D, deterministic=False) -> int:
    return int(load().fa_bwd_workspace_size(B, H, Hk, Sq, Sk, D, int(bool(deterministic))))


def bwd_workspace_size_dv(B, H, Hk, Sq, Sk, D, Dv, deterministic=False) -> int:
    return int(load().fa_bwd_workspace_size_dv(B, H, Hk, Sq, Sk, D, Dv, int(bool(deterministic))))


def alloc_bwd_workspace(q: torch.Tensor, k: torch.Tensor, deterministic=False,
                        v: torch.Tensor | None = None) -> torch.Tensor:
    """Workspace for fa_bwd on these inputs (v: only needed when its head dim differs)."""
    B, Sq, H, D = q.shape
    Sk, Hk = k.shape[1], k.shape[2]
    Dv = v.shape[3] if v is not None else D
    n = bwd_workspace_size_dv(B, H, Hk, Sq, Sk, D, Dv, deterministic)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=q.device)


def fa_fwd(q, k, v, out, lse, softmax_scale, causal=False, window_left=-1, window_right=-1,
           softcap=0.0, stream=None):
    """Writes O into `out` and natural-log LSE into `lse` (C call `fa_fwd`)."""
    lib = load()
    tv = [tensor_view(x) for x in (q, k, v, out, lse)]
    st = lib.fa_fwd(*[ctypes.byref(x) for x in tv], float(softmax_scale), int(bool(causal)),
                    int(window_left), int(window_right), float(softcap), None, 0,
                    _stream_ptr(stream))
    _check(st, "fa_fwd")


def fa_bwd(dout, q, k, v, out, lse, dq, dk, dv, softmax_scale, causal=False, window_left=-1,
           window_right=-1, softcap=0.0, deterministic=False, workspace=None, stream=None):
    """Writes dQ, dK, dV in place (C call `fa_bwd`).  Returns the workspace used."""
    lib = load()
    if workspace is None:
        workspace = alloc_bwd_workspace(q, k, deterministic, v)
    tv = [tensor_view(x) for x in (dout, q, k, v, out, lse, dq, dk, dv)]
    st = lib.fa_bwd(*[ctypes.byref(x) for x in tv], float(softmax_scale), int(bool(causal)),
                    int(window_left), int(window_right), float(softcap), int(bool(deterministic)),
                    ctypes.c_void_p(workspace.data_ptr()), workspace.numel(), _stream_ptr(stream))
    _check(st, "fa_bwd")
    return workspace


def fa_bwd_status(workspace, stream=None) -> int:
    """Device status word of the last fa_bwd on `workspace` (0 = every wait completed)."""
    lib = load()
    out = ctypes.c_int(0)
    st = lib.fa_bwd_status(ctypes.c_void_p(workspace.data_ptr()), _stream_ptr(stream),
                           ctypes.byref(out))
    _check(st, "fa_bwd_status")
    return int(out.value)


ALGO_SPLIT = 0
ALGO_FUSED = 1
ALGO_AUTO = 2


def set_algorithm(algo: int):
    """Backward algorithm for later fa_bwd calls: ALGO_SPLIT (dK/dV kernel + dQ kernel, no
    atomics), ALGO_FUSED (one kernel, fp32 dQ accumulator, ordered when deterministic) or
    ALGO_AUTO (the default: split for deterministic batched bf16 square causal calls, fused
    otherwise)."""
    _check(load().fa_bwd_set_algorithm(int(algo)), "fa_bwd_set_algorithm")


def get_algorithm() -> int:
    return int(load().fa_bwd_get_algorithm())


def set_wait_limit(cycles: int):
    _check(load().fa_debug_set_wait_limit(int(cycles)), "fa_debug_set_wait_limit")


def poison_ordering(enable: bool):
    _check(load().fa_debug_poison_ordering(int(bool(enable))), "fa_debug_poison_ordering")


def profile_enable(enable: bool = True):
    """Record CUDA events around the three backward kernels of every later fa_bwd."""
    _check(load().fa_profile_enable(int(bool(enable))), "fa_profile_enable")


def profile_read():
    """(preprocess_ms, main_ms, convert_ms) of the most recent fa_bwd (waits for it)."""
    ms = (ctypes.c_float * 3)()
    _check(load().fa_profile_read(ms), "fa_profile_read")
    return float(ms[0]), float(ms[1]), float(ms[2])


def fa_bwd_noalloc(dout, q, k, v, out, lse, dq, dk, dv, softmax_scale, causal=False,
                   window_left=-1, window_right=-1, softcap=0.0, deterministic=False,
                   stream=None):
    """C call `fa_bwd_noalloc`: the backward with the library's own fixed scratch (for
    callers that cannot allocate device memory); raises FaError on a non-zero status."""
    lib = load()
    tv = [tensor_view(x) for x in (dout, q, k, v, out, lse, dq, dk, dv)]
    st = lib.fa_bwd_noalloc(*[ctypes.byref(x) for x in tv], float(softmax_scale), int(bool(causal)),
            int(window_left), int(window_right), float(softcap), int(bool(deterministic)),
            _stream_ptr(stream))
    _check(st, "fa_bwd_noalloc")


def fa_bwd_noalloc_status(stream=None) -> int:
    """C call `fa_bwd_noalloc_status`: device status word of the last fa_bwd_noalloc on the
    current device (0 = every bounded wait completed), read and cleared."""
    out = ctypes.c_int(0)
    _check(load().fa_bwd_noalloc_status(_stream_ptr(stream), ctypes.byref(out)),
           "fa_bwd_noalloc_status")
    return int(out.value)


# ------------------------------------------------------------------ packed sequences

def _offsets(cu):
    if cu.dtype != torch.int32 or not cu.is_cuda or cu.dim() != 1:
        raise ValueError("cu_seqlens must be a 1-D int32 CUDA tensor")
    return ctypes.c_void_p(cu.data_ptr())


def _used(used, batch):
    """Optional per-sequence used lengths (seqused_q / seqused_k): None or a 1-D int32 CUDA
    tensor of `batch` entries."""
    if used is None:
        return None
    if used.dtype != torch.int32 or not used.is_cuda or used.dim() != 1 or used.numel() != batch:
        raise ValueError(f"seqused must be a 1-D int32 CUDA tensor of {batch} entries")
    return ctypes.c_void_p(used.data_ptr())


def fa_fwd_varlen(q, k, v, out, lse, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k,
                  softmax_scale, causal=False, window_left=-1, window_right=-1, softcap=0.0,
                  stream=None, seqused_q=None, seqused_k=None):
    """C call `fa_fwd_varlen`: q, out (total_q, H, D), k, v (total_k, Hk, D), lse (H, total_q)."""
    lib = load()
    batch = cu_seqlens_q.numel() - 1
    tv = [tensor_view(x) for x in (q, k, v, out, lse)]
    st = lib.fa_fwd_varlen(*[ctypes.byref(x) for x in tv], _offsets(cu_seqlens_q),
                           _offsets(cu_seqlens_k), _used(seqused_q, batch), _used(seqused_k, batch),
                           batch, int(max_seqlen_q),
                           int(max_seqlen_k), float(softmax_scale), int(bool(causal)),
                           int(window_left), int(window_right), float(softcap), None, 0,
                           _stream_ptr(stream))
    _check(st, "fa_fwd_varlen")


def bwd_varlen_workspace_size(batch, H, total_q, D, deterministic=False) -> int:
    return int(load().fa_bwd_varlen_workspace_size(batch, H, total_q, D, int(bool(deterministic))))


def fa_bwd_varlen(dout, q, k, v, out, lse, dq, dk, dv, cu_seqlens_q, cu_seqlens_k, max_seqlen_q,
                  max_seqlen_k, softmax_scale, causal=False, window_left=-1, window_right=-1,
                  softcap=0.0, deterministic=False, workspace=None, stream=None, seqused_q=None,
                  seqused_k=None):
    """C call `fa_bwd_varlen` (dq, dk, dv written in place).  Returns the workspace used."""
    lib = load()
    batch = cu_seqlens_q.numel() - 1
    if workspace is None:
        n = bwd_varlen_workspace_size(batch, q.shape[1], q.shape[0], q.shape[2], deterministic)
        workspace = torch.empty(max(n, 256), dtype=torch.uint8, device=q.device)
    tv = [tensor_view(x) for x in (dout, q, k, v, out, lse, dq, dk, dv)]
    st = lib.fa_bwd_varlen(*[ctypes.byref(x) for x in tv], _offsets(cu_seqlens_q),
                           _offsets(cu_seqlens_k), _used(seqused_q, batch), _used(seqused_k, batch),
                           batch, int(max_seqlen_q), int(max_seqlen_k),
                           float(softmax_scale), int(bool(causal)), int(window_left),
                           int(window_right), float(softcap), int(bool(deterministic)),
                           ctypes.c_void_p(workspace.data_ptr()), workspace.numel(),
                           _stream_ptr(stream))
    _check(st, "fa_bwd_varlen")
    return workspace


# ------------------------------------------------------------------ block sparsity

def _block_mask_ptr(bm, q, k):
    B, Sq, H = q.shape[0], q.shape[1], q.shape[2]
    Sk = k.shape[1]
    want = (B, H, -(-Sq // 128), -(-Sk // 128))
    if bm.dtype != torch.uint8 or not bm.is_cuda or tuple(bm.shape) != want or not bm.is_contiguous():
        raise ValueError(f"block_mask must be a contiguous uint8 CUDA tensor of shape {want}")
    return ctypes.c_void_p(bm.data_ptr())


def fa_fwd_blocksparse(q, k, v, out, lse, block_mask, softmax_scale, causal=False, window_left=-1,
                       window_right=-1, softcap=0.0, stream=None):
    """C call `fa_fwd_blocksparse` (block_mask: uint8 (B, H, ceil(Sq/128), ceil(Sk/128)))."""
    lib = load()
    tv = [tensor_view(x) for x in (q, k, v, out, lse)]
    st = lib.fa_fwd_blocksparse(*[ctypes.byref(x) for x in tv], _block_mask_ptr(block_mask, q, k),
                                float(softmax_scale), int(bool(causal)), int(window_left),
                                int(window_right), float(softcap), None, 0, _stream_ptr(stream))
    _check(st, "fa_fwd_blocksparse")


def bwd_blocksparse_workspace_size(B, H, Hk, Sq, Sk, D) -> int:
    return int(load().fa_bwd_blocksparse_workspace_size(B, H, Hk, Sq, Sk, D))


def fa_bwd_blocksparse(dout, q, k, v, out, lse, dq, dk, dv, block_mask, softmax_scale, causal=False,
                       window_left=-1, window_right=-1, softcap=0.0, workspace=None, stream=None,
                       deterministic=False):
    """C call `fa_bwd_blocksparse` (dq, dk, dv written in place).  Returns the workspace."""
    lib = load()
    if workspace is None:
        B, Sq, H, D = q.shape
        n = bwd_blocksparse_workspace_size(B, H, k.shape[2], Sq, k.shape[1], D)
        workspace = torch.empty(max(n, 256), dtype=torch.uint8, device=q.device)
    tv = [tensor_view(x) for x in (dout, q, k, v, out, lse, dq, dk, dv)]
    st = lib.fa_bwd_blocksparse(*[ctypes.byref(x) for x in tv], _block_mask_ptr(block_mask, q, k),
                                float(softmax_scale), int(bool(causal)), int(window_left),
                                int(window_right), float(softcap), int(bool(deterministic)),
                                ctypes.c_void_p(workspace.data_ptr()), workspace.numel(),
                                _stream_ptr(stream))
    _check(st, "fa_bwd_blocksparse")
    return workspace

"""GB300-native FlashAttention-2 forward: the Python binding of ``libfa.so``.

The binding only marshals arguments: every step of the computation runs in
the library's CUDA kernels (C ABI in ``include/fa.h``).  PyTorch supplies
device memory and the current stream.  There is no CPU or PyTorch fallback:
if the library is missing, every call raises.

    O, LSE = fwd(Q, K, V, scale=None, is_causal=False)

Q: [B, H, N_q, d], K: [B, H_kv, N_k, d], V: [B, H_kv, N_k, d_v] CUDA tensors
(bf16 or fp32; any strides with a contiguous last dim; H_kv divides H; d_v
may differ from d).  O has Q's dtype and V's head dim, LSE is fp32
[B, H, N_q] (natural log).  The default scale is 1/sqrt(d), as in "Extend
Thunder with CUDA-Python" (flash_attention_reference) and "Blackwell Attention
Example" (blackwell_attention).

Also: ``bwd`` (dQ, dK, dV), ``attention`` (autograd), ``fwd_varlen`` (packed
sequences of different lengths), ``fwd_noalloc``, ``fwd_grouped``, ``axial``
and ``axial_block``; ``sdpa`` routes torch's scaled_dot_product_attention here.
"""
from __future__ import annotations

import ctypes
import math
import threading
from pathlib import Path

import torch

__all__ = ["fwd", "fwd_noalloc", "fwd_varlen", "bwd", "attention", "axial_block", "fwd_grouped", "axial", "check", "debug_set", "FaError", "lib", "build",
           "LIB_PATH", "FA_OK", "FA_ERR_INVALID_ARG", "FA_ERR_UNSUPPORTED", "FA_ERR_CUDA",
           "FA_ERR_TIMEOUT"]

LIB_PATH = Path(__file__).resolve().parent / "_build" / "libfa.so"

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_TIMEOUT = 0, 1, 2, 3, 4
FA_BF16, FA_FP32 = 0, 1
# size of the fixed per-device scratch of fwd_noalloc (FA_SPLITKV_NOALLOC_SCRATCH_BYTES)
SPLITKV_NOALLOC_SCRATCH_BYTES = 128 << 20


class FaTensor(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("stride", ctypes.c_int64 * 4)]


class FaProblem(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("H", ctypes.c_int64), ("N_q", ctypes.c_int64),
                ("N_k", ctypes.c_int64), ("d", ctypes.c_int64),
                ("Q", FaTensor), ("K", FaTensor), ("V", FaTensor), ("O", FaTensor),
                ("LSE", ctypes.c_void_p), ("lse_stride", ctypes.c_int64 * 3),
                ("scale", ctypes.c_float), ("is_causal", ctypes.c_int), ("H_kv", ctypes.c_int64),
                ("Dv", ctypes.c_int64)]


class AxialWeights(ctypes.Structure):
    _fields_ = [("norm_w", ctypes.c_void_p), ("norm_b", ctypes.c_void_p), ("qkv_w", ctypes.c_void_p),
                ("out_w", ctypes.c_void_p), ("out_b", ctypes.c_void_p)]


class FaError(RuntimeError):
    """A non-OK status from libfa.so."""

    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


_lock = threading.Lock()
_lib = None


def build(force: bool = False, ptxas_verbose: bool = False) -> Path:
    """Compile libfa.so for sm_103a (nvcc) into this package's _build/."""
    from ._build import build as _b
    return _b(force=force, ptxas_verbose=ptxas_verbose)


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not LIB_PATH.exists():
                raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                                   "attention_fa2_fwd_02_gb300.build() (no fallback exists)")
            L = ctypes.CDLL(str(LIB_PATH))
            P = ctypes.POINTER
            L.fa_fwd.restype = ctypes.c_int
            L.fa_fwd.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                 ctypes.c_int64, ctypes.c_int64, P(FaTensor), P(FaTensor),
                                 P(FaTensor), ctypes.c_float, ctypes.c_int, P(FaTensor),
                                 ctypes.c_void_p, P(ctypes.c_int64), ctypes.c_void_p]
            L.fa_fwd_grouped.restype = ctypes.c_int
            L.fa_fwd_grouped.argtypes = [ctypes.c_int, ctypes.c_int, P(FaProblem), ctypes.c_void_p]
            L.fa_check.restype = ctypes.c_int
            L.fa_check.argtypes = [ctypes.c_void_p]
            L.fa_status_string.restype = ctypes.c_char_p
            L.fa_status_string.argtypes = [ctypes.c_int]
            L.fa_last_error.restype = ctypes.c_char_p
            L.fa_last_error.argtypes = []
            L.fa_debug_set.restype = None
            L.fa_debug_set.argtypes = [ctypes.c_uint64, ctypes.c_int]
            L.fa_version.restype = ctypes.c_int
            L.fa_version.argtypes = []
            L.fa_fwd_splitkv_workspace_bytes.restype = ctypes.c_size_t
            L.fa_fwd_splitkv_workspace_bytes.argtypes = [ctypes.c_int64] * 4 + [ctypes.c_int]
            L.fa_fwd_splitkv_choose.restype = ctypes.c_int
            L.fa_fwd_splitkv_choose.argtypes = [ctypes.c_int] + [ctypes.c_int64] * 5 + [ctypes.c_int]
            L.fa_fwd_splitkv.restype = ctypes.c_int
            L.fa_fwd_splitkv.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                         ctypes.c_int64, ctypes.c_int64, P(FaTensor), P(FaTensor),
                                         P(FaTensor), ctypes.c_float, ctypes.c_int, P(FaTensor),
                                         ctypes.c_void_p, P(ctypes.c_int64), ctypes.c_int,
                                         ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
            L.fa_fwd_splitkv_noalloc.restype = ctypes.c_int
            L.fa_fwd_splitkv_noalloc.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                                 ctypes.c_int64, ctypes.c_int64, P(FaTensor), P(FaTensor),
                                                 P(FaTensor), ctypes.c_float, ctypes.c_int, P(FaTensor),
                                                 ctypes.c_void_p, P(ctypes.c_int64), ctypes.c_int,
                                                 ctypes.c_void_p]
            L.fa_axial_block_fwd.restype = ctypes.c_int
            L.fa_axial_block_fwd.argtypes = [ctypes.c_int64] * 5 + [ctypes.c_void_p, P(AxialWeights),
                                                                   P(AxialWeights), ctypes.c_void_p, ctypes.c_void_p]
            L.fa_fwd_ws_bytes.restype = ctypes.c_size_t
            L.fa_fwd_ws_bytes.argtypes = [ctypes.c_int] + [ctypes.c_int64] * 6
            L.fa_fwd_ws.restype = ctypes.c_int
            L.fa_fwd_ws.argtypes = [ctypes.c_int] + [ctypes.c_int64] * 6 + [P(FaTensor)] * 3 + \
                [ctypes.c_float, ctypes.c_int, P(FaTensor), ctypes.c_void_p, P(ctypes.c_int64), ctypes.c_void_p,
                 ctypes.c_size_t, ctypes.c_void_p]
            L.fa_fwd_gqa.restype = ctypes.c_int
            L.fa_fwd_gqa.argtypes = [ctypes.c_int] + [ctypes.c_int64] * 6 + [P(FaTensor)] * 3 + \
                [ctypes.c_float, ctypes.c_int, P(FaTensor), ctypes.c_void_p, P(ctypes.c_int64), ctypes.c_void_p]
            L.fa_bwd_gqa.restype = ctypes.c_int
            L.fa_bwd_gqa.argtypes = ([ctypes.c_int] + [ctypes.c_int64] * 6 + [P(FaTensor)] * 5 +
                                     [ctypes.c_void_p, P(ctypes.c_int64), ctypes.c_float, ctypes.c_int] +
                                     [P(FaTensor)] * 3 + [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p])
            L.fa_fwd_varlen.restype = ctypes.c_int
            L.fa_fwd_varlen.argtypes = ([ctypes.c_int] + [ctypes.c_int64] * 8 + [ctypes.c_void_p] * 2 +
                                        [P(FaTensor)] * 3 + [ctypes.c_float, ctypes.c_int, P(FaTensor),
                                                             ctypes.c_void_p, P(ctypes.c_int64), ctypes.c_void_p])
            L.fa_bwd_dv.restype = ctypes.c_int
            L.fa_bwd_dv.argtypes = ([ctypes.c_int] + [ctypes.c_int64] * 7 + [P(FaTensor)] * 5 +
                                    [ctypes.c_void_p, P(ctypes.c_int64), ctypes.c_float, ctypes.c_int] +
                                    [P(FaTensor)] * 3 + [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p])
            L.fa_bwd_workspace_bytes.restype = ctypes.c_size_t
            L.fa_bwd_workspace_bytes.argtypes = [ctypes.c_int64] * 4
            L.fa_bwd.restype = ctypes.c_int
            L.fa_bwd.argtypes = ([ctypes.c_int] + [ctypes.c_int64] * 5 + [P(FaTensor)] * 5 +
                                 [ctypes.c_void_p, P(ctypes.c_int64), ctypes.c_float, ctypes.c_int] +
                                 [P(FaTensor)] * 3 + [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p])
            _lib = L
    return _lib


def _raise_on(status: int) -> None:
    if status != FA_OK:
        L = lib()
        msg = L.fa_last_error().decode()
        raise FaError(status, f"{L.fa_status_string(status).decode()}: {msg}")


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return FA_BF16
    if t.dtype == torch.float32:
        return FA_FP32
    raise TypeError(f"unsupported dtype {t.dtype} (bf16 or fp32)")


def _as4(t: torch.Tensor) -> torch.Tensor:
    if t.dim() == 4:
        return t
    if t.dim() == 3:
        return t.unsqueeze(0)
    if t.dim() == 2:
        return t.unsqueeze(0).unsqueeze(0)
    raise ValueError(f"expected a 2-, 3- or 4-D tensor, got {tuple(t.shape)}")


def _ft(t: torch.Tensor) -> FaTensor:
    s = t.stride()
    return FaTensor(ctypes.c_void_p(t.data_ptr()), (ctypes.c_int64 * 4)(*s))


def _stream_ptr(device: torch.device, stream=None) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def causal_code(is_causal) -> int:
    """The C ABI's is_causal: False -> 0 (no mask), True or "top_left" -> 1,
    "bottom_right" -> 2 (key j visible to query row i iff j <= i + N_k - N_q)."""
    if isinstance(is_causal, str):
        codes = {"top_left": 1, "bottom_right": 2, "none": 0}
        if is_causal not in codes:
            raise ValueError(f"is_causal must be a bool, 'top_left' or 'bottom_right', not {is_causal!r}")
        return codes[is_causal]
    return 1 if is_causal else 0


def _problem(Q, K, V, scale, is_causal, out, lse, with_lse):
    if not (Q.is_cuda and K.is_cuda and V.is_cuda):
        raise ValueError("Q, K, V must be CUDA tensors (this library has no CPU path)")
    if not (Q.dtype == K.dtype == V.dtype):
        raise TypeError("Q, K, V must share one dtype")
    if not (Q.device == K.device == V.device):
        raise ValueError("Q, K, V must be on one device")
    q4, k4, v4 = _as4(Q), _as4(K), _as4(V)
    B, H, N_q, d = q4.shape
    if k4.shape[:3] != v4.shape[:3] or k4.shape[0] != B or k4.shape[3] != d or H % k4.shape[1] != 0:
        raise ValueError(f"shape mismatch: Q{tuple(Q.shape)} K{tuple(K.shape)} V{tuple(V.shape)} "
                         "(K/V heads must divide the query heads)")
    N_k = k4.shape[2]
    d_v = v4.shape[3]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o_shape = (*Q.shape[:-1], d_v)
    if out is None:
        out = torch.empty(o_shape, dtype=Q.dtype, device=Q.device)
    o4 = _as4(out)
    if tuple(out.shape) != o_shape or out.dtype != Q.dtype or out.device != Q.device:
        raise ValueError("out must have Q's leading shape and V's head dim, Q's dtype and device")
    if with_lse and lse is None:
        lse = torch.empty(Q.shape[:-1], dtype=torch.float32, device=Q.device)
    pb = FaProblem()
    pb.B, pb.H, pb.N_q, pb.N_k, pb.d = B, H, N_q, N_k, d
    pb.H_kv = k4.shape[1]
    pb.Dv = d_v
    pb.Q, pb.K, pb.V, pb.O = _ft(q4), _ft(k4), _ft(v4), _ft(o4)
    if lse is not None:
        if lse.dtype != torch.float32 or lse.device != Q.device or lse.shape != Q.shape[:-1]:
            raise ValueError("lse must be fp32 with Q's leading shape, on Q's device")
        l3 = lse
        while l3.dim() < 3:
            l3 = l3.unsqueeze(0)
        pb.LSE = ctypes.c_void_p(l3.data_ptr())
        pb.lse_stride = (ctypes.c_int64 * 3)(*l3.stride())
    else:
        pb.LSE = None
        pb.lse_stride = (ctypes.c_int64 * 3)(0, 0, 0)
    pb.scale = float(scale)
    pb.is_causal = causal_code(is_causal)
    return pb, out, lse


def fwd(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, scale: float | None = None,
        is_causal: bool = False, out: torch.Tensor | None = None,
        lse: torch.Tensor | None = None, with_lse: bool = True, stream=None,
        split_kv: int | None = None, workspace: torch.Tensor | None = None):
    """O, LSE = softmax(scale * Q K^T) V and its log-sum-exp, on the GPU.

    Asynchronous on the current (or given) stream.  Returns (O, LSE); LSE is
    None when ``with_lse`` is False and no ``lse`` buffer is passed.
    ``split_kv``: key-range splits (None = the library's choice for this
    device; 1 = never split).  A split run needs scratch memory, and so does
    an fp32 run whose V tiles are each read by several query tiles (V^T is
    written there once, fa_fwd_ws): ``workspace`` (a CUDA uint8 tensor of at
    least the required bytes) or, if None, one allocated here from PyTorch's
    allocator.
    """
    pb, out, lse = _problem(Q, K, V, scale, is_causal, out, lse, with_lse)
    L = lib()
    code = _dtype_code(Q)
    with torch.cuda.device(Q.device):
        lse_stride = (ctypes.c_int64 * 3)(*pb.lse_stride)
        n_split = 1
        if pb.d in (64, 128) and pb.H_kv == pb.H and pb.Dv == pb.d:  # (split-KV: K/V with the query heads, Dv = d)
            n_split = (L.fa_fwd_splitkv_choose(code, pb.B, pb.H, pb.N_q, pb.N_k, pb.d, pb.is_causal)
                       if split_kv is None else int(split_kv))
        def scratch(need):
            nonlocal workspace
            if workspace is None:
                workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=Q.device)
            if workspace.device != Q.device or workspace.numel() * workspace.element_size() < need:
                raise ValueError(f"workspace must be a CUDA buffer of >= {need} bytes on Q's device")
            return ctypes.c_void_p(workspace.data_ptr()), workspace.numel() * workspace.element_size()

        if pb.Dv != pb.d:  # V with a head dim of its own: the one-problem grouped entry
            st = L.fa_fwd_grouped(code, 1, ctypes.byref(pb), _stream_ptr(Q.device, stream))
        elif n_split == 1:
            need = L.fa_fwd_ws_bytes(code, pb.B, pb.H, pb.H_kv, pb.N_q, pb.N_k, pb.d)
            if need > 0:  # fp32: V^T written once into the workspace
                ws, ws_bytes = scratch(need)
                st = L.fa_fwd_ws(code, pb.B, pb.H, pb.H_kv, pb.N_q, pb.N_k, pb.d,
                                 ctypes.byref(pb.Q), ctypes.byref(pb.K), ctypes.byref(pb.V),
                                 pb.scale, pb.is_causal, ctypes.byref(pb.O), pb.LSE, lse_stride,
                                 ws, ws_bytes, _stream_ptr(Q.device, stream))
            else:
                st = L.fa_fwd_gqa(code, pb.B, pb.H, pb.H_kv, pb.N_q, pb.N_k, pb.d,
                                  ctypes.byref(pb.Q), ctypes.byref(pb.K), ctypes.byref(pb.V),
                                  pb.scale, pb.is_causal, ctypes.byref(pb.O), pb.LSE, lse_stride,
                                  _stream_ptr(Q.device, stream))
        else:
            ws, ws_bytes = scratch(L.fa_fwd_splitkv_workspace_bytes(pb.B, pb.H, pb.N_q, pb.d, n_split))
            st = L.fa_fwd_splitkv(code, pb.B, pb.H, pb.N_q, pb.N_k, pb.d,
                                  ctypes.byref(pb.Q), ctypes.byref(pb.K), ctypes.byref(pb.V),
                                  pb.scale, pb.is_causal, ctypes.byref(pb.O), pb.LSE, lse_stride,
                                  n_split, ws, ws_bytes, _stream_ptr(Q.device, stream))
    _raise_on(st)
    return out, lse


def fwd_noalloc(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, out: torch.Tensor,
                lse: torch.Tensor | None = None, scale: float | None = None, is_causal: bool = False,
                split_kv: int | None = None, stream=None):
    """``fwd`` through fa_fwd_splitkv_noalloc: no device memory is allocated.

    For callers that must not allocate on this path (no allocator of their
    own, or cudaMalloc/cudaFree not allowed where they would synchronise the
    device or could fail).  ``out`` (and ``lse``, if wanted) must be given;
    the split-KV scratch is the library's fixed per-device buffer
    (FA_SPLITKV_NOALLOC_SCRATCH_BYTES), so calls that overlap on the device
    race, and a problem too large for it raises FaError.  Make the first call
    on a device before any stream capture on it.  Returns (out, lse).
    """
    if out is None:
        raise ValueError("fwd_noalloc needs a caller-provided out tensor (it allocates nothing)")
    pb, out, lse = _problem(Q, K, V, scale, is_causal, out, lse, with_lse=False)
    L = lib()
    code = _dtype_code(Q)
    with torch.cuda.device(Q.device):
        if pb.H_kv != pb.H or pb.Dv != pb.d:  # grouped K/V heads or Dv != d: the unsplit kernel (no scratch)
            st = L.fa_fwd_grouped(code, 1, ctypes.byref(pb), _stream_ptr(Q.device, stream))
            _raise_on(st)
            return out, lse
        n_split = 1
        if pb.d in (64, 128):
            n_split = (L.fa_fwd_splitkv_choose(code, pb.B, pb.H, pb.N_q, pb.N_k, pb.d, pb.is_causal)
                       if split_kv is None else int(split_kv))
        st = L.fa_fwd_splitkv_noalloc(code, pb.B, pb.H, pb.N_q, pb.N_k, pb.d,
                                      ctypes.byref(pb.Q), ctypes.byref(pb.K), ctypes.byref(pb.V),
                                      pb.scale, pb.is_causal, ctypes.byref(pb.O), pb.LSE,
                                      (ctypes.c_int64 * 3)(*pb.lse_stride), n_split,
                                      _stream_ptr(Q.device, stream))
    _raise_on(st)
    return out, lse


def fwd_varlen(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cu_seqlens_q: torch.Tensor,
               cu_seqlens_k: torch.Tensor, max_seqlen_q: int, scale: float | None = None,
               is_causal=False, out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
               with_lse: bool = True, stream=None):
    """Attention over a packed batch of sequences of different lengths.

    q: [total_q, H, d], k: [total_k, H_kv, d], v: [total_k, H_kv, d_v] (H_kv
    divides H; d_v may differ from d), bf16, d and d_v multiples of 8 up to
    128, rows of sequence b at cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1
    (and likewise for the keys); the offsets are int32 CUDA tensors of B + 1
    entries from 0 to total.  Each sequence attends only to itself;
    ``is_causal`` (False, True / "top_left", "bottom_right") applies per
    sequence.  ``max_seqlen_q`` bounds the query lengths (it sizes the grid).
    Returns (out [total_q, H, d_v], lse [H, total_q] fp32 or None).
    """
    if not (q.is_cuda and k.is_cuda and v.is_cuda and cu_seqlens_q.is_cuda and cu_seqlens_k.is_cuda):
        raise ValueError("q, k, v and the offsets must be CUDA tensors (this library has no CPU path)")
    if q.dim() != 3 or k.dim() != 3 or v.dim() != 3 or k.shape[:2] != v.shape[:2] or k.shape[2] != q.shape[2]:
        raise ValueError(f"expected q [total_q, H, d], k [total_k, H_kv, d], v [total_k, H_kv, d_v]: "
                         f"{tuple(q.shape)} {tuple(k.shape)} {tuple(v.shape)}")
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k, v must share one dtype")
    for name, cu in (("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_k", cu_seqlens_k)):
        if cu.dtype != torch.int32 or cu.dim() != 1 or not cu.is_contiguous() or cu.device != q.device:
            raise ValueError(f"{name} must be a contiguous 1-D int32 tensor on q's device")
    if cu_seqlens_q.numel() != cu_seqlens_k.numel() or cu_seqlens_q.numel() < 2:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must both hold B + 1 >= 2 offsets")
    total_q, H, d = q.shape
    total_k, H_kv = k.shape[0], k.shape[1]
    B = cu_seqlens_q.numel() - 1
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o_shape = (total_q, H, v.shape[2])
    if out is None:
        out = torch.empty(o_shape, dtype=q.dtype, device=q.device)
    if out.shape != o_shape or out.dtype != q.dtype or out.device != q.device:
        raise ValueError("out must be [total_q, H, d_v] in q's dtype, on q's device")
    if with_lse and lse is None:
        lse = torch.empty((H, total_q), dtype=torch.float32, device=q.device)
    if lse is not None and (lse.shape != (H, total_q) or lse.dtype != torch.float32 or lse.device != q.device):
        raise ValueError("lse must be fp32 [H, total_q] on q's device")

    def view(t):  # [total, heads, d] -> [1, heads, total, d]
        return _ft(t.permute(1, 0, 2).unsqueeze(0))
    tq, tk, tv, to = view(q), view(k), view(v), view(out)
    lse_stride = (ctypes.c_int64 * 3)(0, *(lse.stride() if lse is not None else (0, 0)))
    L = lib()
    with torch.cuda.device(q.device):
        st = L.fa_fwd_varlen(_dtype_code(q), B, H, H_kv, total_q, total_k, int(max_seqlen_q), d, v.shape[2],
                             ctypes.c_void_p(cu_seqlens_q.data_ptr()), ctypes.c_void_p(cu_seqlens_k.data_ptr()),
                             ctypes.byref(tq), ctypes.byref(tk), ctypes.byref(tv), float(scale),
                             causal_code(is_causal), ctypes.byref(to),
                             ctypes.c_void_p(lse.data_ptr()) if lse is not None else None, lse_stride,
                             _stream_ptr(q.device, stream))
    _raise_on(st)
    return out, lse


def bwd(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, O: torch.Tensor, LSE: torch.Tensor,
        dO: torch.Tensor, scale: float | None = None, is_causal: bool = False,
        dQ: torch.Tensor | None = None, dK: torch.Tensor | None = None, dV: torch.Tensor | None = None,
        workspace: torch.Tensor | None = None, stream=None):
    """(dQ, dK, dV) of sum(dO * O) for O, LSE = fwd(Q, K, V, scale, is_causal).

    bf16 tensors; Q, K (and dQ, dK) of head dim d, V, O, dO (and dV) of head
    dim d_v (= d unless V has its own), both multiples of 8 up to 128; LSE
    fp32 as ``fwd`` returns it.  Missing outputs and the scratch
    ``workspace`` (a CUDA uint8 tensor of fa_bwd_workspace_bytes(B, H, N_q,
    max(d, d_v))) are allocated here from PyTorch's allocator.  Asynchronous
    on the current (or given) stream.
    """
    if not all(t.is_cuda for t in (Q, K, V, O, LSE, dO)):
        raise ValueError("Q, K, V, O, LSE, dO must be CUDA tensors (this library has no CPU path)")
    q4, k4, v4, o4, g4 = _as4(Q), _as4(K), _as4(V), _as4(O), _as4(dO)
    B, H, N_q, d = q4.shape
    N_k = k4.shape[2]
    d_v = v4.shape[3]
    if o4.shape[:3] != q4.shape[:3] or o4.shape[3] != d_v or g4.shape != o4.shape or \
            v4.shape[:3] != k4.shape[:3] or k4.shape[0] != B or H % k4.shape[1] != 0 or k4.shape[3] != d:
        raise ValueError("shape mismatch between Q, K, V, O and dO (K/V heads must divide the query heads; "
                         "V, O, dO share their head dim)")
    H_kv = k4.shape[1]
    if LSE.dtype != torch.float32 or LSE.shape != Q.shape[:-1]:
        raise ValueError("LSE must be fp32 with Q's leading shape")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dQ = torch.empty_like(Q) if dQ is None else dQ
    dK = torch.empty_like(K) if dK is None else dK
    dV = torch.empty_like(V) if dV is None else dV
    for name, t, ref in (("dQ", dQ, Q), ("dK", dK, K), ("dV", dV, V)):
        if t.shape != ref.shape or t.dtype != ref.dtype or t.device != ref.device:
            raise ValueError(f"{name} must match the shape, dtype and device of its input")
    L = lib()
    need = L.fa_bwd_workspace_bytes(B, H, N_q, max(d, d_v))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=Q.device)
    if workspace.device != Q.device or workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"workspace must be a CUDA buffer of >= {need} bytes on Q's device")
    l3 = LSE
    while l3.dim() < 3:
        l3 = l3.unsqueeze(0)
    with torch.cuda.device(Q.device):
        st = L.fa_bwd_dv(_dtype_code(Q), B, H, H_kv, N_q, N_k, d, d_v,
                      ctypes.byref(_ft(q4)), ctypes.byref(_ft(k4)), ctypes.byref(_ft(v4)), ctypes.byref(_ft(o4)),
                      ctypes.byref(_ft(g4)), ctypes.c_void_p(l3.data_ptr()), (ctypes.c_int64 * 3)(*l3.stride()),
                      float(scale), causal_code(is_causal),
                      ctypes.byref(_ft(_as4(dQ))), ctypes.byref(_ft(_as4(dK))), ctypes.byref(_ft(_as4(dV))),
                      ctypes.c_void_p(workspace.data_ptr()), workspace.numel() * workspace.element_size(),
                      _stream_ptr(Q.device, stream))
    _raise_on(st)
    return dQ, dK, dV


class _Attention(torch.autograd.Function):
    """Autograd wrapper: forward through fa_fwd, backward through fa_bwd."""

    @staticmethod
    def forward(ctx, Q, K, V, scale, is_causal):
        O, LSE = fwd(Q, K, V, scale=scale, is_causal=is_causal)
        ctx.save_for_backward(Q, K, V, O, LSE)
        ctx.scale, ctx.is_causal = scale, is_causal
        return O

    @staticmethod
    def backward(ctx, dO):
        Q, K, V, O, LSE = ctx.saved_tensors
        dQ, dK, dV = bwd(Q, K, V, O, LSE, dO.contiguous(), scale=ctx.scale, is_causal=ctx.is_causal)
        return dQ, dK, dV, None, None


def attention(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, scale: float | None = None,
              is_causal: bool | str = False) -> torch.Tensor:
    """softmax(scale * Q K^T) V with autograd: forward and backward on the GPU.
    is_causal: False, True / "top_left", or "bottom_right"."""
    if scale is None:
        scale = 1.0 / math.sqrt(Q.shape[-1])
    return _Attention.apply(Q, K, V, float(scale), is_causal if isinstance(is_causal, str) else bool(is_causal))


def axial_block(x: torch.Tensor, row: dict, col: dict, heads: int = 4, out: torch.Tensor | None = None,
                stream=None) -> torch.Tensor:
    """The axial attention block (row pass, then column pass), fused per sequence.

    x: contiguous fp32 CUDA tensor [B, H, W, D] (D = 64, heads = 4, H, W <= 32).
    row / col: dicts of CUDA fp32 tensors norm_w, norm_b [D], qkv_w [3D, D],
    out_w [D, D], out_b [D] (nn.LayerNorm / nn.Linear parameter layouts).
    Returns out (allocated if not given; may be x for an in-place update).
    """
    if not x.is_cuda or x.dtype != torch.float32 or x.dim() != 4 or not x.is_contiguous():
        raise ValueError("x must be a contiguous fp32 CUDA tensor [B, H, W, D]")
    out = torch.empty_like(x) if out is None else out
    if out.shape != x.shape or out.dtype != x.dtype or out.device != x.device or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor like x")
    keep = []

    def pack(p):
        ts = [p[k].contiguous() for k in ("norm_w", "norm_b", "qkv_w", "out_w", "out_b")]
        for t in ts:
            if not t.is_cuda or t.dtype != torch.float32:
                raise ValueError("axial block weights must be fp32 CUDA tensors")
        keep.extend(ts)
        return AxialWeights(*(ctypes.c_void_p(t.data_ptr()) for t in ts))
    rw, cw = pack(row), pack(col)
    B, H, W, D = x.shape
    with torch.cuda.device(x.device):
        st = lib().fa_axial_block_fwd(B, H, W, D, heads, ctypes.c_void_p(x.data_ptr()), ctypes.byref(rw),
                                      ctypes.byref(cw), ctypes.c_void_p(out.data_ptr()), _stream_ptr(x.device, stream))
    _raise_on(st)
    return out


def fwd_grouped(problems, stream=None):
    """Several independent problems in as few launches as possible.

    ``problems``: list of dicts with keys Q, K, V and optional scale,
    is_causal, out, lse, with_lse.  Returns a list of (O, LSE).
    """
    if not problems:
        return []
    built, results = [], []
    for pr in problems:
        pb, out, lse = _problem(pr["Q"], pr["K"], pr["V"], pr.get("scale"),
                                pr.get("is_causal", False), pr.get("out"), pr.get("lse"),
                                pr.get("with_lse", True))
        built.append(pb)
        results.append((out, lse))
    dt = _dtype_code(problems[0]["Q"])
    if any(_dtype_code(p["Q"]) != dt for p in problems):
        raise TypeError("all problems of a grouped call share one dtype")
    dev = problems[0]["Q"].device
    arr = (FaProblem * len(built))(*built)
    with torch.cuda.device(dev):
        st = lib().fa_fwd_grouped(dt, len(built), arr, _stream_ptr(dev, stream))
    _raise_on(st)
    return results


def axial(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, scale: float | None = None,
          with_lse: bool = False, stream=None):
    """Row and column attention over an axial grid, in one launch.

    Q, K, V: [B, Hg, Wg, heads, hd] tensors (contiguous).  Row attention runs
    along Wg for every (b, hg, head); column attention along Hg for every
    (b, wg, head).  Both read the inputs in place through strided views.
    Returns ((O_row, LSE_row), (O_col, LSE_col)), O_* shaped like Q.
    """
    B, Hg, Wg, nh, hd = Q.shape

    # .view (never .reshape): the views must alias the tensors, no copies
    def row_view(x):  # [B*Hg, heads, Wg, (hd)]
        return x.permute(0, 1, 3, 2, *range(4, x.dim())).view(B * Hg, nh, Wg, *x.shape[4:])

    def col_view(x):  # [B, Wg*heads, Hg, (hd)]
        return x.permute(0, 2, 3, 1, *range(4, x.dim())).view(B, Wg * nh, Hg, *x.shape[4:])

    O_row = torch.empty_like(Q)
    O_col = torch.empty_like(Q)
    lse_row = torch.empty((B, Hg, Wg, nh), dtype=torch.float32, device=Q.device) if with_lse else None
    lse_col = torch.empty((B, Hg, Wg, nh), dtype=torch.float32, device=Q.device) if with_lse else None
    probs = [
        dict(Q=row_view(Q), K=row_view(K), V=row_view(V), scale=scale, out=row_view(O_row),
             lse=None if lse_row is None else row_view(lse_row), with_lse=with_lse),
        dict(Q=col_view(Q), K=col_view(K), V=col_view(V), scale=scale, out=col_view(O_col),
             lse=None if lse_col is None else col_view(lse_col), with_lse=with_lse),
    ]
    fwd_grouped(probs, stream=stream)
    return (O_row, lse_row), (O_col, lse_col)


def check(stream=None, device=None) -> None:
    """Synchronise and raise FaError if a kernel's bounded wait expired."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        st = lib().fa_check(_stream_ptr(dev, stream))
    _raise_on(st)


def debug_set(timeout_ns: int = 0, flags: int = 0) -> None:
    """Test hooks: device wait limit (0 = default 1 s) and fault-injection flags."""
    lib().fa_debug_set(int(timeout_ns), int(flags))

"""fp64 CPU attention oracle -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never does, and
this package imports nothing from the product package: the two share no code.

The arithmetic lives in ``attention_oracle.c`` (plain C, fp64, untiled; its
header states the definition and the passages it follows).  This module only
compiles that file with gcc, loads it with ctypes and loops over the leading
(batch, head) dimensions.

Reading of the pages it encodes ("Extend Thunder with CUDA-Python",
flash_attention_reference; "Blackwell Attention Example", kernel docstring):

* O = softmax(scale * Q K^T) V per (batch, head) slice, SDPA layout [..., N, d];
* LSE = log sum_j exp(s_ij), natural log of the scaled scores;
* causal: key j visible to query row i iff j <= i (top-left alignment,
  is_causal = True or 1); bottom-right alignment (is_causal = 2): j <= i +
  N_k - N_q, a row that sees no key has O = 0 and LSE = -inf;
* backward ("Blackwell Attention Example", section "Backward Kernel
  Implementation"): the gradients of sum(dO * O) with respect to Q, K and V,
  with delta_i = dO_i . O_i and dS = P (dP - delta).
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "attention_oracle.c"
_LIB_PATH = _HERE / "_build" / "liboracle.so"
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> Path:
    """Compile ``attention_oracle.c`` into ``oracle/_build/liboracle.so``."""
    _LIB_PATH.parent.mkdir(parents=True, exist_ok=True)
    if (not force and _LIB_PATH.exists()
            and _LIB_PATH.stat().st_mtime >= _SRC.stat().st_mtime):
        return _LIB_PATH
    tmp = _LIB_PATH.with_suffix(f".so.tmp{os.getpid()}")
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
           str(_SRC), "-o", str(tmp), "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(str(build()))
            f = lib.oracle_attention_slice_v
            f.restype = ctypes.c_int
            f.argtypes = [
                ctypes.c_void_p, ctypes.c_int64,
                ctypes.c_void_p, ctypes.c_int64,
                ctypes.c_void_p, ctypes.c_int64,
                ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                ctypes.c_double, ctypes.c_int,
                ctypes.c_void_p, ctypes.c_int64,
                ctypes.c_void_p, ctypes.c_void_p,
            ]
            lib.oracle_num_threads.restype = ctypes.c_int
            g = lib.oracle_attention_bwd_slice_v
            g.restype = ctypes.c_int
            g.argtypes = [
                ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64,
                ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64,
                ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                ctypes.c_double, ctypes.c_int,
                ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
            ]
            _lib = lib
    return _lib


def num_threads() -> int:
    """Host threads the oracle's parallel loop uses."""
    return int(_load().oracle_num_threads())


def _as_f32(x) -> np.ndarray:
    if hasattr(x, "detach"):  # a torch tensor (bf16 widens exactly to fp32)
        x = x.detach().cpu().float().numpy()
    x = np.asarray(x)
    if x.dtype != np.float32:
        x32 = x.astype(np.float32)
        if not np.array_equal(x32.astype(x.dtype), x):
            raise ValueError("oracle inputs must be exactly representable in fp32")
        x = x32
    return x


def _causal_code(is_causal) -> int:
    """False/0 none, True/1 top-left, 2 or "bottom_right" bottom-right."""
    if is_causal == "bottom_right":
        return 2
    if is_causal in (2,) and not isinstance(is_causal, bool):
        return 2
    return 1 if is_causal else 0


def attention(Q, K, V, scale: float, is_causal: bool = False, rows=None):
    """fp64 attention of every (batch..., head) slice.

    Q: [..., N_q, d]; K: [..., N_k, d]; V: [..., N_k, d_v] with the same
    leading dims (d_v may differ from d: "Blackwell Attention Example",
    blackwell_attention).
    rows: optional 1-D sequence of query rows to evaluate in every slice.
    Returns (O, LSE) as float64 numpy arrays [..., n_rows, d_v] and [..., n_rows].
    """
    Q, K, V = _as_f32(Q), _as_f32(K), _as_f32(V)
    if Q.ndim < 2 or K.shape[:-1] != V.shape[:-1] or K.ndim != V.ndim or Q.shape[:-2] != K.shape[:-2] \
            or Q.shape[-1] != K.shape[-1]:
        raise ValueError(f"bad shapes Q{Q.shape} K{K.shape} V{V.shape}")
    lead = Q.shape[:-2]
    N_q, d = Q.shape[-2:]
    N_k = K.shape[-2]
    d_v = V.shape[-1]
    if rows is None:
        rows_arr = None
        n_rows = N_q
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
        n_rows = rows_arr.size
    Qs = np.ascontiguousarray(Q.reshape(-1, N_q, d))
    Ks = np.ascontiguousarray(K.reshape(-1, N_k, d))
    Vs = np.ascontiguousarray(V.reshape(-1, N_k, d_v))
    O = np.empty((Qs.shape[0], n_rows, d_v), dtype=np.float64)
    L = np.empty((Qs.shape[0], n_rows), dtype=np.float64)
    lib = _load()
    rows_ptr = None if rows_arr is None else rows_arr.ctypes.data
    for s in range(Qs.shape[0]):
        rc = lib.oracle_attention_slice_v(
            Qs[s].ctypes.data, d, Ks[s].ctypes.data, d, Vs[s].ctypes.data, d_v,
            N_q, N_k, d, d_v, float(scale), _causal_code(is_causal),
            rows_ptr, n_rows, O[s].ctypes.data, L[s].ctypes.data)
        if rc != 0:
            raise RuntimeError(f"oracle_attention_slice_v failed with {rc}")
    return O.reshape(*lead, n_rows, d_v), L.reshape(*lead, n_rows)


def attention_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, scale: float, is_causal=False):
    """fp64 attention of a packed batch of sequences of different lengths.

    q: [total_q, H, d], k: [total_k, H, d], v: [total_k, H, d_v]; sequence b holds the packed
    rows cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 of q (and the same for k, v
    with cu_seqlens_k) and attends to its own keys only: the definition applied
    to each sequence as its own [H, len, d] problem (the causal alignment, too,
    is per sequence).  Returns (O [total_q, H, d_v], LSE [H, total_q]) float64.
    """
    q, k, v = _as_f32(q), _as_f32(k), _as_f32(v)
    cq = [int(x) for x in np.asarray(cu_seqlens_q).reshape(-1)]
    ck = [int(x) for x in np.asarray(cu_seqlens_k).reshape(-1)]
    if q.ndim != 3 or v.ndim != 3 or k.shape[:2] != v.shape[:2] or k.shape[1:] != q.shape[1:] or len(cq) != len(ck) \
            or cq[0] != 0 or ck[0] != 0 or cq[-1] != q.shape[0] or ck[-1] != k.shape[0]:
        raise ValueError("bad packed shapes or offsets")
    total_q, H, d = q.shape
    O = np.zeros((total_q, H, v.shape[2]), dtype=np.float64)
    L = np.full((H, total_q), -np.inf, dtype=np.float64)
    for b in range(len(cq) - 1):
        q0, q1, k0, k1 = cq[b], cq[b + 1], ck[b], ck[b + 1]
        if q1 < q0 or k1 < k0:
            raise ValueError("offsets must not decrease")
        if q1 == q0:
            continue
        if k1 == k0:  # a sequence without keys: every row sees none
            continue
        Ob, Lb = attention(q[q0:q1].transpose(1, 0, 2), k[k0:k1].transpose(1, 0, 2),
                           v[k0:k1].transpose(1, 0, 2), scale, is_causal)
        O[q0:q1] = Ob.transpose(1, 0, 2)
        L[:, q0:q1] = Lb
    return O, L


def attention_bwd(Q, K, V, dO, scale: float, is_causal: bool = False, q_rows=None, k_rows=None):
    """fp64 gradients (dQ, dK, dV) of sum(dO * O) for every (batch..., head) slice.

    Q: [..., N_q, d]; K: [..., N_k, d]; V: [..., N_k, d_v]; dO: [..., N_q, d_v]
    (d_v may differ from d).  q_rows / k_rows: optional 1-D sequences of query
    / key rows to evaluate in every slice (default all).  Returns float64 numpy
    arrays dQ [..., n_q_rows, d], dK [..., n_k_rows, d], dV [..., n_k_rows, d_v].
    """
    Q, K, V, dO = _as_f32(Q), _as_f32(K), _as_f32(V), _as_f32(dO)
    if Q.ndim < 2 or K.ndim != V.ndim or Q.ndim != dO.ndim or K.shape[:-1] != V.shape[:-1] \
            or Q.shape[:-1] != dO.shape[:-1] or Q.shape[:-2] != K.shape[:-2] or Q.shape[-1] != K.shape[-1] \
            or dO.shape[-1] != V.shape[-1]:
        raise ValueError(f"bad shapes Q{Q.shape} K{K.shape} V{V.shape} dO{dO.shape}")
    lead = Q.shape[:-2]
    N_q, d = Q.shape[-2:]
    N_k = K.shape[-2]
    d_v = V.shape[-1]

    def rows_of(rows, n):
        if rows is None:
            return None, n
        a = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
        return a, a.size
    qr, nq = rows_of(q_rows, N_q)
    kr, nk = rows_of(k_rows, N_k)
    Qs = np.ascontiguousarray(Q.reshape(-1, N_q, d))
    Gs = np.ascontiguousarray(dO.reshape(-1, N_q, d_v))
    Ks = np.ascontiguousarray(K.reshape(-1, N_k, d))
    Vs = np.ascontiguousarray(V.reshape(-1, N_k, d_v))
    dQ = np.empty((Qs.shape[0], nq, d), dtype=np.float64)
    dK = np.empty((Qs.shape[0], nk, d), dtype=np.float64)
    dV = np.empty((Qs.shape[0], nk, d_v), dtype=np.float64)
    lib = _load()
    for s in range(Qs.shape[0]):
        rc = lib.oracle_attention_bwd_slice_v(
            Qs[s].ctypes.data, d, Ks[s].ctypes.data, d, Vs[s].ctypes.data, d_v, Gs[s].ctypes.data, d_v,
            N_q, N_k, d, d_v, float(scale), _causal_code(is_causal),
            None if qr is None else qr.ctypes.data, nq, None if kr is None else kr.ctypes.data, nk,
            dQ[s].ctypes.data, dK[s].ctypes.data, dV[s].ctypes.data)
        if rc != 0:
            raise RuntimeError(f"oracle_attention_bwd_slice_v failed with {rc}")
    return dQ.reshape(*lead, nq, d), dK.reshape(*lead, nk, d), dV.reshape(*lead, nk, d_v)


def layer_norm(x, weight, bias, eps: float = 1e-5):
    """fp64 LayerNorm over the last dim: (x - mean) / sqrt(var + eps) * w + b,
    var the biased (population) variance, as torch.nn.LayerNorm."""
    x = np.asarray(x, dtype=np.float64)
    mean = x.mean(-1, keepdims=True)
    var = ((x - mean) ** 2).mean(-1, keepdims=True)
    return (x - mean) / np.sqrt(var + eps) * np.asarray(weight, np.float64) + np.asarray(bias, np.float64)


def _axial_pass(seqs, p, heads: int):
    """One pass of the axial block on sequences [S, L, D] (fp64): the axial
    transcript's _attn_ref (LayerNorm, bias-free QKV projection, per-head
    softmax(q k^T / sqrt(d)) v, output projection with bias) plus the
    residual of its forward."""
    S, L, D = seqs.shape
    d = D // heads
    xn = layer_norm(seqs, p["norm_w"], p["norm_b"])
    qkv = xn @ np.asarray(p["qkv_w"], np.float64).T            # [S, L, 3D]
    qkv = qkv.reshape(S, L, 3, heads, d)
    q, k, v = (qkv[:, :, i].transpose(0, 2, 1, 3) for i in range(3))   # [S, heads, L, d]
    # softmax(q k^T / sqrt(d)) v per (sequence, head), fp64, written out
    sc = (q @ k.transpose(0, 1, 3, 2)) / math.sqrt(d)                  # [S, heads, L, L]
    pr = np.exp(sc - sc.max(-1, keepdims=True))
    pr /= pr.sum(-1, keepdims=True)
    o = (pr @ v).transpose(0, 2, 1, 3).reshape(S, L, D)
    return seqs + o @ np.asarray(p["out_w"], np.float64).T + np.asarray(p["out_b"], np.float64)


def axial_block(x, row, col, heads: int):
    """fp64 forward of the axial attention block on x [B, H, W, D]: the row
    pass over the W-long rows, then the column pass over the H-long columns of
    the updated grid ("axial attention" transcript, the module's forward).
    row / col: dicts of norm_w, norm_b [D], qkv_w [3D, D], out_w [D, D],
    out_b [D].  Returns float64 [B, H, W, D]."""
    x = np.asarray(x, dtype=np.float64)
    B, H, W, D = x.shape
    y = _axial_pass(x.reshape(B * H, W, D), row, heads).reshape(B, H, W, D)
    yc = y.transpose(0, 2, 1, 3).reshape(B * W, H, D)
    return _axial_pass(yc, col, heads).reshape(B, W, H, D).transpose(0, 2, 1, 3)

"""Routing of PyTorch's scaled_dot_product_attention to this library.

"Extend Thunder with CUDA-Python" (section "Running our kernel in Thunder")
registers a flash-attention kernel as the implementation of the SDPA symbol
when the call has no mask and no dropout; this module is the same idea for
plain PyTorch:

* ``scaled_dot_product_attention`` has the signature of
  ``torch.nn.functional.scaled_dot_product_attention`` and computes it with
  fa_fwd / fa_bwd (autograd included).  Arguments the library does not
  implement (an explicit mask, dropout) raise ``NotImplementedError``: there
  is no fallback to another implementation.
* The forward and backward are registered as ``torch.library`` custom ops
  (``fa_gb300::fwd`` / ``fa_gb300::bwd``) with shape functions, so that the
  call can sit inside ``torch.compile``d code as an opaque op.
* ``routed()`` is a context manager that replaces
  ``torch.nn.functional.scaled_dot_product_attention`` by this function for
  the duration of a block (and restores it afterwards, also on exceptions).
"""
from __future__ import annotations

import contextlib
import math

import torch

from . import bwd as _bwd
from . import fwd as _fwd

__all__ = ["scaled_dot_product_attention", "routed"]


@torch.library.custom_op("fa_gb300::fwd", mutates_args=())
def _fwd_op(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: float,
            is_causal: bool) -> tuple[torch.Tensor, torch.Tensor]:
    o, lse = _fwd(q, k, v, scale=scale, is_causal=is_causal)
    return o, lse


@_fwd_op.register_fake
def _(q, k, v, scale, is_causal):
    return q.new_empty((*q.shape[:-1], v.shape[-1])), q.new_empty(q.shape[:-1], dtype=torch.float32)


@torch.library.custom_op("fa_gb300::bwd", mutates_args=())
def _bwd_op(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor, lse: torch.Tensor,
            do: torch.Tensor, scale: float, is_causal: bool) -> tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    dq, dk, dv = _bwd(q, k, v, o, lse, do.contiguous(), scale=scale, is_causal=is_causal)
    return dq, dk, dv


@_bwd_op.register_fake
def _(q, k, v, o, lse, do, scale, is_causal):
    return torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)


def _setup_context(ctx, inputs, output):
    q, k, v, scale, is_causal = inputs
    o, lse = output
    # the backward below gives the gradients of O only: a gradient reaching
    # LSE would be dropped, so autograd is told that LSE has none
    ctx.mark_non_differentiable(lse)
    ctx.save_for_backward(q, k, v, o, lse)
    ctx.scale, ctx.is_causal = scale, is_causal


def _backward(ctx, do, dlse):
    q, k, v, o, lse = ctx.saved_tensors
    dq, dk, dv = _bwd_op(q, k, v, o, lse, do, ctx.scale, ctx.is_causal)
    return dq, dk, dv, None, None


torch.library.register_autograd("fa_gb300::fwd", _backward, setup_context=_setup_context)


def scaled_dot_product_attention(query: torch.Tensor, key: torch.Tensor, value: torch.Tensor,
                                 attn_mask: torch.Tensor | None = None, dropout_p: float = 0.0,
                                 is_causal: bool = False, scale: float | None = None,
                                 enable_gqa: bool = False) -> torch.Tensor:
    """``torch.nn.functional.scaled_dot_product_attention`` on this library.

    query [..., H, N_q, d], key [..., H_kv, N_k, d], value [..., H_kv, N_k, d_v]
    (H_kv = H unless ``enable_gqa``, then H_kv must divide H; d_v may differ
    from d, as in PyTorch).  The causal mask is the top-left one, as in
    PyTorch.  bf16 or fp32; the head dims and layouts fa_fwd supports (the
    backward: bf16, d and d_v multiples of 8 up to 128).
    """
    if attn_mask is not None:
        raise NotImplementedError("attn_mask is not supported (only is_causal)")
    if dropout_p != 0.0:
        raise NotImplementedError("dropout is not supported")
    if query.dim() < 2 or key.dim() != query.dim() or value.dim() != key.dim() or value.shape[:-1] != key.shape[:-1]:
        raise ValueError("query, key, value must share their rank; key and value all but their last dim")
    if query.dim() >= 3 and key.shape[-3] != query.shape[-3] and not enable_gqa:
        raise ValueError("query and key/value head counts differ: pass enable_gqa=True")
    if scale is None:
        scale = 1.0 / math.sqrt(query.shape[-1])
    lead = query.shape[:-3] if query.dim() > 4 else None
    if lead is not None:  # fold extra leading dims into the batch
        query = query.reshape(-1, *query.shape[-3:])
        key = key.reshape(-1, *key.shape[-3:])
        value = value.reshape(-1, *value.shape[-3:])
    o, _ = _fwd_op(query, key, value, float(scale), bool(is_causal))
    return o if lead is None else o.reshape(*lead, *o.shape[-3:])


@contextlib.contextmanager
def routed():
    """Within the block, torch.nn.functional.scaled_dot_product_attention is
    this module's function."""
    import torch.nn.functional as F
    orig = F.scaled_dot_product_attention
    F.scaled_dot_product_attention = scaled_dot_product_attention
    try:
        yield
    finally:
        F.scaled_dot_product_attention = orig

"""The product path has no CPU or PyTorch fallback: without the built library
every call raises, and CPU tensors are refused before any computation (CPU
only; no GPU needed)."""
from __future__ import annotations

import pytest
import torch

import attention_fa2_fwd_02_gb300 as fa
from attention_fa2_fwd_02_gb300 import sdpa


@pytest.fixture
def no_library(tmp_path, monkeypatch):
    monkeypatch.setattr(fa, "LIB_PATH", tmp_path / "missing" / "libfa.so")
    monkeypatch.setattr(fa, "_lib", None)
    yield


def test_missing_library_raises(no_library):
    with pytest.raises(RuntimeError, match="no fallback"):
        fa.lib()
    with pytest.raises(RuntimeError):
        fa.check()


def _cpu(*shape, dtype=torch.bfloat16):
    return torch.zeros(shape, dtype=dtype)


def test_cpu_tensors_are_refused():
    q = _cpu(1, 2, 64, 128)
    with pytest.raises(ValueError, match="CUDA"):
        fa.fwd(q, q, q)
    with pytest.raises(ValueError, match="CUDA"):
        fa.bwd(q, q, q, q, _cpu(1, 2, 64, dtype=torch.float32), q)
    cu = torch.tensor([0, 64], dtype=torch.int32)
    p = _cpu(64, 2, 128)
    with pytest.raises(ValueError, match="CUDA"):
        fa.fwd_varlen(p, p, p, cu, cu, 64)
    with pytest.raises(ValueError, match="CUDA"):
        fa.attention(q, q, q)


def test_sdpa_rejects_what_it_does_not_implement():
    q = _cpu(1, 2, 16, 64)
    with pytest.raises(NotImplementedError):
        sdpa.scaled_dot_product_attention(q, q, q, attn_mask=torch.ones(16, 16, dtype=torch.bool))
    with pytest.raises(NotImplementedError):
        sdpa.scaled_dot_product_attention(q, q, q, dropout_p=0.1)

"""The fused axial attention block (fa_axial_block_fwd) against the fp64 block
oracle on the same seeded inputs and weights.  Tolerance (fp32 arithmetic,
LayerNorm, sums of 64 and 192 terms, fast exp in the softmax): max-abs error
<= 2e-4 * (1 + max|ref|)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import attention_fa2_fwd_02_gb300 as fa
from attention_fa2_fwd_02_gb300.inputs import AXIAL_BLOCK, AxialBlockWorkload, normal

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa.build()
    yield


def _cuda(p):
    return {k: v.cuda() for k, v in p.items()}


def _check(got, ref, what):
    g = got.cpu().numpy()
    assert np.isfinite(g).all(), what
    err = float(np.abs(g - ref).max())
    assert err <= 2e-4 * (1.0 + float(np.abs(ref).max())), f"{what}: max|err|={err:.3e}"


@pytest.mark.parametrize("shape", [(4, 32, 32), (2, 5, 7), (1, 32, 1), (3, 1, 32), (1, 1, 1), (2, 17, 31)])
def test_axial_block_matches_oracle(oracle_mod, shape):
    B, H, W = shape
    w = AxialBlockWorkload(B=B, H=H, W=W, seed=20 + B + H + W)
    x, row, col = w.make()
    y = fa.axial_block(x.cuda(), _cuda(row), _cuda(col))
    fa.check()
    ref = oracle_mod.axial_block(x.numpy(), {k: v.numpy() for k, v in row.items()},
                                 {k: v.numpy() for k, v in col.items()}, 4)
    _check(y, ref, f"shape {shape}")


def test_axial_block_in_place(oracle_mod):
    x, row, col = AXIAL_BLOCK.make()
    xd = x.cuda()
    out = fa.axial_block(xd, _cuda(row), _cuda(col), out=xd)
    fa.check()
    assert out.data_ptr() == xd.data_ptr()
    ref = oracle_mod.axial_block(x.numpy(), {k: v.numpy() for k, v in row.items()},
                                 {k: v.numpy() for k, v in col.items()}, 4)
    _check(xd, ref, "in place")


def test_axial_block_rejects_unsupported():
    x = torch.zeros(1, 4, 40, 64, device="cuda")
    _, row, col = AXIAL_BLOCK.make()
    with pytest.raises(fa.FaError):
        fa.axial_block(x, _cuda(row), _cuda(col))      # W > 32
    with pytest.raises(fa.FaError):
        fa.axial_block(torch.zeros(1, 4, 4, 64, device="cuda"), _cuda(row), _cuda(col), heads=2)

"""Bounded waits of every tensor-core kernel: the test hook (fa_debug_set
flag 1) makes block 0's load warp withhold one tile, so the waits on it run
out within the short limit set here.  The launch then ends with every role
out of its loop and its copies and MMAs drained, fa_check reports
FA_ERR_TIMEOUT (and clears the error word), and the next launch on the same
context is correct against the oracle.  No GPU fault, trap or hang is
involved: a wait that gives up only returns.

Kernels covered: the two-stage forward (bf16; plain, split-KV and packed
variable-length instantiations), the single-stage forward (bf16 d = 256;
fp32 d = 128 and 64 both with V^T from the workspace and with the in-kernel
V transpose; fp32 split-KV) and the backward.
"""
from __future__ import annotations

import ctypes
import math

import numpy as np
import pytest
import torch

import attention_fa2_fwd_02_gb300 as fa
from attention_fa2_fwd_02_gb300.inputs import normal, packed, qkv

pytestmark = pytest.mark.gpu

TOL = {torch.bfloat16: (2e-2, 1e-2), torch.float32: (3e-3, 2e-3)}
LIMIT_NS = 50_000_000  # 50 ms


@pytest.fixture(scope="module", autouse=True)
def _setup(oracle_mod):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa.build()
    fa.debug_set(0, 0)
    yield
    fa.debug_set(0, 0)


def _times_out(launch):
    """Run `launch` with one tile withheld; it must end with FA_ERR_TIMEOUT."""
    fa.debug_set(LIMIT_NS, 1)
    try:
        launch()
        with pytest.raises(fa.FaError) as ei:
            fa.check()
        assert ei.value.status == fa.FA_ERR_TIMEOUT
    finally:
        fa.debug_set(0, 0)
    fa.check()  # the error word was cleared, the context still works


def _close(O, L, O_ref, L_ref, dtype, what):
    to, tl = TOL[dtype]
    O, L = O.float().cpu().numpy(), L.cpu().numpy()
    assert np.isfinite(O).all() and np.isfinite(L).all(), what
    eo, el = float(np.abs(O - O_ref).max()), float(np.abs(L - L_ref).max())
    assert eo <= to and el <= tl, f"{what}: max|dO|={eo:.3e} max|dLSE|={el:.3e}"


def _fwd_no_workspace(Q, K, V, scale, causal, out, lse):
    """fa_fwd_gqa straight through the C ABI: for fp32, the in-kernel V
    transpose (the binding would pass a workspace and take the V^T pass)."""
    pb, out, lse = fa._problem(Q, K, V, scale, causal, out, lse, True)
    st = fa.lib().fa_fwd_gqa(fa._dtype_code(Q), pb.B, pb.H, pb.H_kv, pb.N_q, pb.N_k, pb.d, ctypes.byref(pb.Q),
                             ctypes.byref(pb.K), ctypes.byref(pb.V), pb.scale, pb.is_causal, ctypes.byref(pb.O),
                             pb.LSE, (ctypes.c_int64 * 3)(*pb.lse_stride), fa._stream_ptr(Q.device))
    fa._raise_on(st)


# (name, dtype, N_q, N_k, d, causal, split, workspace): every case gives block
# 0 a first work unit with at least two key tiles, so the withheld second K
# tile is awaited.  workspace=False calls fa_fwd_gqa (fp32: in-kernel V
# transpose); True goes through the binding (fp32: the V^T pass).
FWD_CASES = [
    ("two_stage_bf16_d128_split", torch.bfloat16, 256, 2048, 128, False, 2, True),
    ("two_stage_bf16_d64_causal", torch.bfloat16, 384, 384, 64, True, 1, True),
    ("single_stage_bf16_d256", torch.bfloat16, 256, 512, 256, False, 1, True),
    ("single_stage_fp32_vt_d128", torch.float32, 256, 512, 128, False, 1, True),
    ("single_stage_fp32_vt_d64_causal", torch.float32, 300, 300, 64, True, 1, True),
    ("single_stage_fp32_d128", torch.float32, 256, 512, 128, False, 1, False),
    ("single_stage_fp32_d64_causal", torch.float32, 300, 300, 64, True, 1, False),
    ("single_stage_fp32_d128_split", torch.float32, 128, 2048, 128, False, 2, True),
]


@pytest.mark.parametrize("case", FWD_CASES, ids=[c[0] for c in FWD_CASES])
def test_forward_withheld_tile_times_out_then_runs_correctly(oracle_mod, case):
    name, dtype, nq, nk, d, causal, split, workspace = case
    Q, K, V = qkv((1, 2, nq, d), (1, 2, nk, d), 91 + d + nk, dtype)
    Qd, Kd, Vd = Q.cuda(), K.cuda(), V.cuda()
    scale = 1 / math.sqrt(d)

    def run(out=None, lse=None):
        if workspace:
            fa.fwd(Qd, Kd, Vd, scale=scale, is_causal=causal, split_kv=split, out=out, lse=lse)
        else:
            _fwd_no_workspace(Qd, Kd, Vd, scale, causal, out, lse)

    _times_out(run)
    O = torch.full(Qd.shape, float("nan"), dtype=dtype, device="cuda")
    L = torch.full(Qd.shape[:-1], float("nan"), dtype=torch.float32, device="cuda")
    run(O, L)
    fa.check()
    O_ref, L_ref = oracle_mod.attention(Q, K, V, scale, causal)
    _close(O, L, O_ref, L_ref, dtype, name)


def test_varlen_withheld_tile_times_out_then_runs_correctly(oracle_mod):
    q, k, v, cu_q, cu_k = packed([300, 200], [400, 260], 2, 2, 128, seed=93)
    qd, kd, vd, cqd, ckd = q.cuda(), k.cuda(), v.cuda(), cu_q.cuda(), cu_k.cuda()
    _times_out(lambda: fa.fwd_varlen(qd, kd, vd, cqd, ckd, 300))
    O, L = fa.fwd_varlen(qd, kd, vd, cqd, ckd, 300)
    fa.check()
    O_ref, L_ref = oracle_mod.attention_varlen(q.float().numpy(), k.float().numpy(), v.float().numpy(),
                                               cu_q.numpy(), cu_k.numpy(), 1 / math.sqrt(128), 0)
    _close(O, L, O_ref, L_ref, torch.bfloat16, "varlen")


def test_backward_withheld_step_times_out_then_runs_correctly(oracle_mod):
    Q, K, V = qkv((1, 2, 512, 128), (1, 2, 384, 128), 95, torch.bfloat16)
    dO = normal((1, 2, 512, 128), 96, torch.bfloat16)
    Qd, Kd, Vd, dOd = Q.cuda(), K.cuda(), V.cuda(), dO.cuda()
    scale = 1 / math.sqrt(128)
    O, L = fa.fwd(Qd, Kd, Vd, scale=scale)
    fa.check()
    _times_out(lambda: fa.bwd(Qd, Kd, Vd, O, L, dOd, scale=scale))
    grads = fa.bwd(Qd, Kd, Vd, O, L, dOd, scale=scale)
    fa.check()
    refs = oracle_mod.attention_bwd(Q, K, V, dO, scale, False)
    for nm, got, ref in zip(("dQ", "dK", "dV"), grads, refs):
        err = float(np.abs(got.float().cpu().numpy() - ref).max())
        assert err <= 1.5e-2 * float(np.abs(ref).max()) + 1e-3, f"{nm}: max|err|={err:.3e}"

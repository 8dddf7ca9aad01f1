"""GPU parity of the log-sum-exp combine alone: oracle partials in, GPU combine out.

The end-to-end tests only feed the combine partials that the split pass wrote,
whose LSEs sit within a few units of each other. Here the fp32 partial O and log2
LSE of every split are drawn directly (seeded), written into a plan's workspace
in its layout ([S][rows][d] fp32 O, then [S][rows] fp32 LSE at the plan's
offset), and folded by mla_split_combine (d_v = 512, with and without the
attention sink) and sdpa_split_combine (d = 128), for every output cast. The
oracle folds the very same fp32 values in fp64 ("The Split-K Dispatch", "The LSE
Combine Strategy"; FlashMLA PR #25, "What changes": the combine owns the sink;
cuDNN-frontend PR #768: an empty split enters as O = 0 / LSE = -inf and the
combine owns the amax of the recombined O).

Adversarial LSE patterns: spreads above 100 (weights far below fp32's range),
a single finite split among empty ones, every split empty (with a sink: O = 0,
LSE = -inf), and up to 64 splits. Tolerances: the parity bar of _gpu_util (fp32
O row-wise 2e-3, LSE 1e-5, casts within one code step / ulp), plus 1e-5
row-wise on the fp32 output, since the combine alone computes in fp32 from fp32
inputs.
"""
import numpy as np
import pytest
import torch

import oracle.mla as om
from _gpu_util import assert_cast_close, assert_lse_close, assert_o_close, check_status
from split_kv_sparse_gb300 import binding as b

pytestmark = pytest.mark.gpu

TORCH_OUT = {"f32": torch.float32, "bf16": torch.bfloat16, "e4m3": torch.uint8}


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "the -m gpu tests need a CUDA GPU"
    b.lib()
    check_status()


def _partials(S, rows, d, pattern, seed):
    """fp32 partials [S, rows, d] and log2 LSEs [S, rows] (as float64 holding fp32 values)."""
    rng = np.random.default_rng(seed)
    O = rng.standard_normal((S, rows, d)).astype(np.float32)
    if pattern == "close":
        L = rng.uniform(-8.0, 8.0, (S, rows))
    elif pattern == "spread":
        # one split per row far above the others (> 100 log2 units), the rest spread widely
        L = rng.uniform(-60.0, 60.0, (S, rows))
        top = rng.integers(0, S, rows)
        L[top, np.arange(rows)] = 110.0 + rng.uniform(0.0, 10.0, rows)
    elif pattern == "single":
        L = np.full((S, rows), -np.inf)
        L[rng.integers(0, S, rows), np.arange(rows)] = rng.uniform(-20.0, 20.0, rows)
    elif pattern == "mixed":
        L = rng.uniform(-30.0, 30.0, (S, rows))
        L[rng.random((S, rows)) < 0.5] = -np.inf
        L[:, :3] = -np.inf                        # rows with every split empty
    else:
        raise ValueError(pattern)
    L = L.astype(np.float32)
    O[np.isneginf(L)] = 0.0                       # an empty split stores O = 0
    return O.astype(np.float64), L.astype(np.float64)


def _workspace(plan, O, L, dev):
    S, rows, d = O.shape
    ws = torch.zeros(plan.workspace_bytes, dtype=torch.uint8, device=dev)
    ws[: S * rows * d * 4].view(torch.float32).copy_(torch.from_numpy(O.astype(np.float32)).reshape(-1))
    off = plan.lse_acc_offset
    ws[off: off + S * rows * 4].view(torch.float32).copy_(torch.from_numpy(L.astype(np.float32)).reshape(-1))
    return ws


def _check(out, lse, amax, O_ref, L_ref, out_dtype, inv_scale):
    if out_dtype == "f32":
        assert_o_close(out.numpy(), O_ref)
        assert_o_close(out.numpy(), O_ref, rtol=1e-5, what="O (combine alone, 1e-5)")
    else:
        assert_cast_close(out, O_ref, out_dtype, inv_scale)
    assert_lse_close(lse, L_ref)
    amax_ref = float(np.max(np.abs(O_ref)))
    assert abs(amax - amax_ref) <= 2e-3 * amax_ref


@pytest.mark.parametrize("out_dtype", ["f32", "bf16", "e4m3"])
@pytest.mark.parametrize("pattern", ["close", "spread", "single", "mixed"])
@pytest.mark.parametrize("S", [2, 3, 16, 17, 64])
@pytest.mark.parametrize("with_sink", [False, True])
def test_mla_combine_alone(S, pattern, out_dtype, with_sink):
    dev = torch.device("cuda")
    s_q = 5
    plan = b.mla_decode_plan(s_q, 640, force_splits=S)
    assert plan.num_splits == S
    O_s, L_s = _partials(S, s_q * 64, 512, pattern, seed=S * 31 + len(pattern))
    sink = np.random.default_rng(S).standard_normal(64).astype(np.float32) if with_sink else None
    if with_sink:
        sink[:4] = -np.inf                      # a -inf sink changes nothing
    O_ref, L_ref = om.combine(O_s.reshape(S, s_q, 64, 512), L_s.reshape(S, s_q, 64),
                              sink=None if sink is None else sink.astype(np.float64))
    inv_scale = 64.0 if out_dtype == "e4m3" else 1.0
    ws = _workspace(plan, O_s, L_s, dev)
    out = torch.empty(s_q, 64, 512, dtype=TORCH_OUT[out_dtype], device=dev)
    lse = torch.empty(s_q, 64, dtype=torch.float32, device=dev)
    amax = torch.full((1,), 123.0, dtype=torch.float32, device=dev)
    sink_d = torch.from_numpy(sink).to(dev) if with_sink else None
    b.mla_split_combine(plan, s_q, ws, sink_d, out_dtype, inv_scale, out, lse, amax)
    torch.cuda.synchronize()
    check_status()
    _check(out.cpu(), lse.cpu().double().numpy(), float(amax.cpu()[0]), O_ref, L_ref, out_dtype, inv_scale)


@pytest.mark.parametrize("out_dtype", ["f32", "bf16", "e4m3"])
@pytest.mark.parametrize("pattern", ["close", "spread", "single", "mixed"])
@pytest.mark.parametrize("S", [2, 5, 16, 64])
def test_dense_combine_alone(S, pattern, out_dtype):
    dev = torch.device("cuda")
    batch, h_q, h_kv, total_q = 3, 32, 8, 7
    plan = b.sdpa_fp8_decode_plan(batch, h_q, h_kv, 128, 4, total_q, 8192, force_splits=S)
    assert plan.num_splits == S
    O_s, L_s = _partials(S, total_q * h_q, 128, pattern, seed=S * 17 + len(pattern))
    O_ref, L_ref = om.combine(O_s.reshape(S, total_q, h_q, 128), L_s.reshape(S, total_q, h_q), sink=None)
    inv_scale = 64.0 if out_dtype == "e4m3" else 1.0
    ws = _workspace(plan, O_s, L_s, dev)
    out = torch.empty(total_q, h_q, 128, dtype=TORCH_OUT[out_dtype], device=dev)
    lse = torch.empty(total_q, h_q, dtype=torch.float32, device=dev)
    amax = torch.full((1,), 123.0, dtype=torch.float32, device=dev)
    b.sdpa_split_combine(plan, total_q, ws, out_dtype, inv_scale, out, lse, amax)
    torch.cuda.synchronize()
    check_status()
    _check(out.cpu(), lse.cpu().double().numpy(), float(amax.cpu()[0]), O_ref, L_ref, out_dtype, inv_scale)

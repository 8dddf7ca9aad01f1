"""The decode kernels' bounded waits, made to run out on the real kernels.

Every pipeline wait of the sparse-MLA decode kernel (uniform schedule with the
direct epilogue or split partials, and the balanced schedule whose cut tokens
leave partials for the combine) and of the dense FP8 kernel gives up after a time limit, records
MLA_STATUS_TIMEOUT and the site of the wait in the status word, and aborts its
CTA: the other roles stop at their next wait, the CTA waits for its own copies
and MMAs in flight, frees its tensor memory and exits. mla_set_wait_limit_ns
shortens that limit to 200 ns here, far below the latency of any row or tile
load, so real waits run out (no flag is withheld and nothing faults). The
test then checks the status, restores the limit, and requires the next
ordinary call on the same context to match the oracle.
"""
import numpy as np
import pytest
import torch

import oracle.sdpa as osd
from _gpu_util import assert_lse_close, assert_o_close, check_status, oracle_mla
from split_kv_sparse_gb300 import binding as b
from split_kv_sparse_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

SHORT_NS = 200


@pytest.fixture(autouse=True)
def _restore_limit():
    assert torch.cuda.is_available(), "the -m gpu tests need a CUDA GPU"
    check_status()
    yield
    b.mla_set_wait_limit_ns(0)


def _mla_call(inp, plan, ws, dev):
    out = torch.full((inp.s_q, 64, 512), float("nan"), device=dev)
    lse = torch.full((inp.s_q, 64), float("nan"), device=dev)
    b.mla_sparse_decode(plan, inp.s_q, inp.q.to(dev), inp.kv.to(dev), inp.n_kv, inp.idx.to(dev), inp.sm_scale,
                        inp.sink.to(dev), "f32", 1.0, out, lse, None, ws)
    return out, lse


def _flush_l2(dev):
    """A 256 MiB write: the next call's first loads come from DRAM, so its first
    waits last far longer than the short limit (inputs just copied to the device
    can otherwise still sit in L2, and a wait that ends within the first polls
    never reads the timer)."""
    torch.empty(256 << 20, dtype=torch.uint8, device=dev).fill_(1)


def _expect_timeout():
    st, site = b.mla_get_status()          # synchronises the device first
    assert st & b.MLA_STATUS_TIMEOUT, f"no timeout recorded (status {st:#x})"
    assert site != 0
    assert b.mla_get_status() == (0, 0)    # read and cleared


@pytest.mark.parametrize("kind,S,num_sms", [("direct", 1, 0), ("split", 3, 0),
                                            ("balanced", b.MLA_FORCE_BALANCED, 3)])
def test_mla_waits_run_out_then_the_next_call_is_correct(kind, S, num_sms):
    dev = torch.device("cuda")
    inp = wl.mla_inputs(2, 32768, 640, seed=500, with_sink=True)
    plan = b.mla_decode_plan(2, 640, force_splits=S, num_sms=num_sms)
    assert (plan.balanced_ctas > 0) == (kind == "balanced")
    ws = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device=dev)
    if plan.workspace_bytes:
        b.mla_workspace_init(plan, ws)
    wsp = ws if plan.workspace_bytes else None
    _flush_l2(dev)
    b.mla_set_wait_limit_ns(SHORT_NS)
    _mla_call(inp, plan, wsp, dev)
    _expect_timeout()
    b.mla_set_wait_limit_ns(0)
    out, lse = _mla_call(inp, plan, wsp, dev)
    torch.cuda.synchronize()
    check_status()
    O, L = oracle_mla(inp)
    assert_o_close(out.cpu().double().numpy(), O)
    assert_lse_close(lse.cpu().double().numpy(), L)


@pytest.mark.parametrize("S", [1, 3])
def test_dense_waits_run_out_then_the_next_call_is_correct(S):
    dev = torch.device("cuda")
    # long sequences: dozens of tiles per CTA, so some of its waits outlast the
    # short limit whatever the timer's granularity
    inp = wl.sdpa_inputs(2, 8, 2, 128, q_per_seq=(1, 3), kv_len=(12000, 16000), seed=501)
    total_q, total_kv = int(inp.cu_seqlens_q[-1]), int(inp.cu_seqlens_kv[-1])
    plan = b.sdpa_fp8_decode_plan(2, 8, 2, 128, 3, total_q, 16000, force_splits=S)
    ws = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device=dev)
    ds = [torch.tensor([x], dtype=torch.float32, device=dev) for x in (inp.descale_q, inp.descale_k, inp.descale_v)]
    args = (inp.q.to(dev), inp.k.to(dev), inp.v.to(dev), inp.cu_seqlens_q.to(dev), inp.cu_seqlens_kv.to(dev))

    def call():
        out = torch.full((total_q, 8, 128), float("nan"), device=dev)
        lse = torch.full((total_q, 8), float("nan"), device=dev)
        b.sdpa_fp8_decode(plan, total_q, total_kv, *args, ds[0], ds[1], ds[2], inp.sm_scale, "f32", 1.0, out, lse,
                          None, ws if plan.workspace_bytes else None)
        return out, lse

    _flush_l2(dev)
    b.mla_set_wait_limit_ns(SHORT_NS)
    call()
    _expect_timeout()
    b.mla_set_wait_limit_ns(0)
    out, lse = call()
    torch.cuda.synchronize()
    check_status()
    O, L = osd.attention(inp)
    assert_o_close(out.cpu().double().numpy(), O)
    assert_lse_close(lse.cpu().double().numpy(), L)


def test_wait_limit_argument_range():
    with pytest.raises(b.SplitKVError):
        b.mla_set_wait_limit_ns(99)
    with pytest.raises(b.SplitKVError):
        b.mla_set_wait_limit_ns(10_000_000_001)
    b.mla_set_wait_limit_ns(0)

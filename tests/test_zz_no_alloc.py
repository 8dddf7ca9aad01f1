"""The decode entry point that allocates nothing (mla_sparse_decode_noalloc).

Some callers of this library cannot call cudaMalloc. One example is a plugin whose
host framework owns all device memory through a fixed plan and hands the plugin
only its input and output buffers. Another is code on a path where an allocation
could block on device synchronisation. For them the split pass keeps its fp32
partial workspace in a 16 MiB array inside the library's own device image.

These tests compare that entry point, called through the C ABI, with the
regular one (mla_sparse_decode with a caller-allocated workspace) and with the
fp64 oracle, on two calls in a row; check that the automatic split count always
fits the array; and check that an oversized forced request is refused. The file
is named so pytest collects it last: a run that stops at its first failure has
already run every other test by the time it gets here.
"""
import numpy as np
import pytest
import torch

from _gpu_util import assert_lse_close, assert_o_close, check_status, oracle_mla
from split_kv_sparse_gb300 import binding as b
from split_kv_sparse_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _regular(inp, S, dev):
    plan = b.mla_decode_plan(inp.s_q, inp.topk, force_splits=S)
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=dev) if plan.workspace_bytes else None
    if ws is not None:
        b.mla_workspace_init(plan, ws)
    out = torch.empty(inp.s_q, 64, 512, dtype=torch.float32, device=dev)
    lse = torch.empty(inp.s_q, 64, dtype=torch.float32, device=dev)
    b.mla_sparse_decode(plan, inp.s_q, inp.q.to(dev), inp.kv.to(dev), inp.n_kv, inp.idx.to(dev), inp.sm_scale,
                        inp.sink.to(dev), "f32", 1.0, out, lse, None, ws)
    return out, lse, plan.num_splits


def _noalloc(inp, S, dev):
    out = torch.full((inp.s_q, 64, 512), float("nan"), device=dev)
    lse = torch.full((inp.s_q, 64), float("nan"), device=dev)
    b.mla_sparse_decode_noalloc(inp.s_q, inp.topk, inp.q.to(dev), inp.kv.to(dev), inp.n_kv, inp.idx.to(dev),
                                inp.sm_scale, inp.sink.to(dev), S, "f32", 1.0, out, lse)
    torch.cuda.synchronize()
    check_status()
    return out, lse


def test_noalloc_matches_the_allocating_entry_point_on_two_calls():
    assert torch.cuda.is_available(), "needs a CUDA GPU"
    dev = torch.device("cuda")
    # two calls in a row with different shapes and split counts: the second one
    # reuses the array the first one left behind
    for s_q, seed, S in [(6, 101, 5), (16, 102, 4)]:
        inp = wl.mla_inputs(s_q, 32768, 640, seed=seed, with_sink=True)
        ref_out, ref_lse, used_S = _regular(inp, S, dev)
        assert used_S > 1            # the split pass (which needs the scratch) runs
        out, lse = _noalloc(inp, S, dev)
        assert_o_close(out.cpu().double().numpy(), ref_out.cpu().double().numpy())
        assert_lse_close(lse.cpu().double().numpy(), ref_lse.cpu().double().numpy())
        O, L = oracle_mla(inp)
        assert_o_close(out.cpu().double().numpy(), O)
        assert_lse_close(lse.cpu().double().numpy(), L)


@pytest.mark.parametrize("s_q", [1, 6, 32])
def test_noalloc_automatic_split_count_fits_the_array(s_q):
    """num_splits = 0: the automatic choice is made among the split counts whose
    workspace fits the array, so an ordinary shape is never refused (s_q = 32 would
    need 16.8 MB with the unbounded choice)."""
    dev = torch.device("cuda")
    inp = wl.mla_inputs(s_q, 32768, 640, seed=200 + s_q, with_sink=True)
    out, lse = _noalloc(inp, 0, dev)
    O, L = oracle_mla(inp)
    assert_o_close(out.cpu().double().numpy(), O)
    assert_lse_close(lse.cpu().double().numpy(), L)


def test_noalloc_refuses_a_workspace_beyond_its_array():
    dev = torch.device("cuda")
    inp = wl.mla_inputs(16, 4096, 640, seed=7, index_mode="uniform")
    out = torch.full((16, 64, 512), 3.0, device=dev)
    # 8 splits x 16 tokens x 64 heads x 513 floats > 16 MiB
    with pytest.raises(b.SplitKVError) as e:
        b.mla_sparse_decode_noalloc(16, 640, inp.q.to(dev), inp.kv.to(dev), inp.n_kv, inp.idx.to(dev),
                                    inp.sm_scale, None, 8, "f32", 1.0, out)
    assert e.value.status == 3
    torch.cuda.synchronize()
    assert torch.all(out == 3.0)     # nothing was launched
    check_status()

"""GPU parity of the one-split grid whose last wave is cut into splits.

With one split per token and more tokens than SMs, the last wave of (token) CTAs
would hold r tokens on r SMs while the rest idle. The plan then cuts those r
tokens into min(num_blocks, num_sms // r) >= 3 splits: the whole tokens write
their rows in the decode kernel, the tail's partials are folded by a combine over
the tail rows only. Every case here checks every token against the fp64 oracle
(or a sample of them on the device's SMs), with the tolerances of _gpu_util.
"""
import numpy as np
import pytest
import torch

from _gpu_util import assert_cast_close, assert_lse_close, assert_o_close, check_status, oracle_mla, run_mla
from split_kv_sparse_gb300 import binding as b
from split_kv_sparse_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "the -m gpu tests need a CUDA GPU"
    b.lib()
    check_status()


def tail_shape(s_q, nblk, sms):
    """(first tail token, splits, dim groups) of the tail rule, or None: restated from
    the header (splits when at least 3 fit, else two dim groups per token when 2 r
    <= SMs)."""
    if s_q <= sms:
        return None
    waves = -(-s_q // sms)
    r = s_q - (waves - 1) * sms
    st = min(nblk, sms // r)
    if st >= 3:
        return (s_q - r, st, 0)
    return (s_q - r, 0, 2) if 2 * r <= sms else None


@pytest.mark.parametrize("s_q,topk,num_sms", [
    (10, 640, 8),     # 2 tail tokens, 4 splits of 3, 3, 2, 2 blocks
    (9, 640, 4),      # three waves, 1 tail token in 4 splits
    (13, 200, 6),     # ragged top-k (4 blocks, the last of 8 rows): 1 tail token, 4 one-block splits
    (21, 640, 10),    # 1 tail token in 10 one-block splits
    (7, 128, 4),      # 2 blocks: 3 tail tokens, too many for two CTAs each -> no tail
    (14, 640, 8),     # 6 tail tokens: 1 split each, 12 CTAs for dims -> no tail
    (11, 640, 8),     # 3 tail tokens: 2 splits would not pay -> two dim groups each
    (12, 640, 8),     # 4 tail tokens on two dim groups each (8 CTAs)
    (9, 200, 6),      # ragged top-k (4 blocks, the last of 8 rows): 3 tail tokens on two dim groups
])
@pytest.mark.parametrize("with_sink", [False, True])
def test_tail_matches_oracle(s_q, topk, num_sms, with_sink):
    inp = wl.mla_inputs(s_q, 32768, topk, seed=500 + s_q * 3 + num_sms, with_sink=with_sink,
                        index_mode="window" if topk >= 128 else "uniform")
    O, L = oracle_mla(inp)
    r = run_mla(inp, 0, num_sms=num_sms)
    plan = r["plan"]
    assert plan.num_splits == 1 and plan.tail_ctas == num_sms
    shape = tail_shape(s_q, plan.num_blocks, num_sms)
    assert (shape is None) == ((s_q, topk, num_sms) in ((7, 128, 4), (14, 640, 8)))
    if (s_q, topk, num_sms) in ((11, 640, 8), (12, 640, 8), (9, 200, 6)):
        assert shape[2] == 2
    assert_o_close(r["out"].numpy(), O)
    assert_lse_close(r["lse"], L)


@pytest.mark.parametrize("s_q", [10, 12])
@pytest.mark.parametrize("out_dtype", ["bf16", "e4m3"])
def test_tail_casts_and_amax(out_dtype, s_q):
    """Whole tokens are cast by the decode kernel and the tail tokens by the combine
    (s_q 10: 4 splits) or by their two dim-group CTAs (s_q 12); the amax covers all."""
    inp = wl.mla_inputs(s_q, 32768, 640, seed=71, v_mean=1.0, with_sink=True)
    O, L = oracle_mla(inp)
    r = run_mla(inp, 0, out_dtype=out_dtype, inv_scale=64.0, with_amax=True, num_sms=8)
    assert tail_shape(s_q, 10, 8) == ((8, 4, 0) if s_q == 10 else (8, 0, 2))
    assert_cast_close(r["out"], O, out_dtype, 64.0)
    assert_lse_close(r["lse"], L)
    assert abs(r["amax"] - float(np.abs(O).max())) <= 2e-3 * float(np.abs(O).max())


def test_tail_amax_from_the_tail():
    """The largest |O| sits in a tail token: only the combine can report it. Token 9
    reads 640 rows of its own, appended to the cache, whose V dims are shifted by 16."""
    inp = wl.mla_inputs(10, 32768, 640, seed=73, with_sink=True)
    extra = inp.kv[:640].clone()
    extra[:, :512] += 16.0
    kv = torch.cat([inp.kv, extra])
    idx = inp.idx.clone()
    idx[9] = torch.arange(32768, 32768 + 640, dtype=idx.dtype)
    inp = wl.MlaInputs(q=inp.q, kv=kv, idx=idx, sink=inp.sink, sm_scale=inp.sm_scale)
    O, L = oracle_mla(inp)
    assert np.abs(O[9]).max() > np.abs(O[:9]).max()
    r = run_mla(inp, 0, out_dtype="bf16", with_amax=True, num_sms=8)
    assert_cast_close(r["out"], O, "bf16")
    assert abs(r["amax"] - float(np.abs(O).max())) <= 2e-3 * float(np.abs(O).max())


def test_tail_padding_and_empty_tokens():
    """An all-padding tail token is O = 0, LSE = -inf; a tail split whose rows are all
    masked drops out of the combine; an all-padding whole token too."""
    inp = wl.mla_inputs(10, 32768, 640, seed=79)
    idx = inp.idx.clone()
    idx[9, :] = -1               # tail token: nothing valid
    idx[8, 0:192] = -1           # tail token 8, split 0 (blocks 0-2): no valid row
    idx[8, 300:310] = 40000      # out of range: masked
    idx[3, :] = -1               # a whole token with nothing valid
    inp = wl.MlaInputs(q=inp.q, kv=inp.kv, idx=idx, sink=None, sm_scale=inp.sm_scale)
    O, L = oracle_mla(inp)
    r = run_mla(inp, 0, num_sms=8)
    assert_o_close(r["out"].numpy(), O)
    assert_lse_close(r["lse"], L)
    assert np.all(np.isneginf(r["lse"][9])) and np.all(r["out"][9].numpy() == 0)


def test_tail_bf16_partials():
    """The tail's partials in bf16 (the plan's opt-in): the same tolerance."""
    inp = wl.mla_inputs(10, 32768, 640, seed=83, with_sink=True)
    O, L = oracle_mla(inp)
    dev = torch.device("cuda")
    plan = b.mla_decode_plan(10, 640, num_sms=8)
    ws32 = plan.workspace_bytes
    b.mla_plan_set_partials_bf16(plan, 1)
    assert 0 < plan.workspace_bytes < ws32
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=dev)
    out = torch.empty(10, 64, 512, dtype=torch.float32, device=dev)
    lse = torch.empty(10, 64, dtype=torch.float32, device=dev)
    b.mla_sparse_decode(plan, 10, inp.q.to(dev), inp.kv.to(dev), inp.n_kv, inp.idx.to(dev), inp.sm_scale,
                        inp.sink.to(dev), "f32", 1.0, out, lse, None, ws)
    torch.cuda.synchronize()
    check_status()
    assert_o_close(out.cpu().numpy(), O)
    assert_lse_close(lse.cpu().double().numpy(), L)


def test_tail_fewer_tokens_than_planned():
    """A plan for 20 tokens on 8 SMs called with 10 (r = 2: 4 splits), 12 (r = 4: two
    dim groups each) and 8 (one wave: no tail): the tail follows the call's s_q."""
    inp = wl.mla_inputs(12, 32768, 640, seed=89)
    dev = torch.device("cuda")
    plan = b.mla_decode_plan(20, 640, num_sms=8)
    assert plan.tail_ctas == 8
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=dev)
    for s_q in (10, 12, 8):
        sub = wl.MlaInputs(q=inp.q[:s_q], kv=inp.kv, idx=inp.idx[:s_q], sink=None, sm_scale=inp.sm_scale)
        O, L = oracle_mla(sub)
        out = torch.empty(s_q, 64, 512, dtype=torch.float32, device=dev)
        lse = torch.empty(s_q, 64, dtype=torch.float32, device=dev)
        b.mla_sparse_decode(plan, s_q, sub.q.to(dev), sub.kv.to(dev), sub.n_kv, sub.idx.to(dev), sub.sm_scale,
                            None, "f32", 1.0, out, lse, None, ws)
        torch.cuda.synchronize()
        check_status()
        assert_o_close(out.cpu().numpy(), O, what=f"O s_q={s_q}")
        assert_lse_close(lse.cpu().double().numpy(), L, what=f"LSE s_q={s_q}")


@pytest.mark.parametrize("s_q", [160, 228, 320])
def test_tail_on_device_sms_sampled(s_q):
    """The automatic plan on the device's SMs: 160 tokens on 152 SMs leave 8 in the
    last wave (cut into one-block splits), 320 leave 16, 228 leave 76 (two dim groups
    each); tokens around the wave edge and the whole tail against the oracle, e4m3
    output as the bench runs it."""
    inp = wl.mla_inputs(s_q, 131072, 640, seed=91 + s_q)
    r = run_mla(inp, 0, out_dtype="e4m3", inv_scale=64.0)
    plan = r["plan"]
    sms = plan.num_sms
    shape = tail_shape(s_q, plan.num_blocks, sms)
    first = shape[0] if shape is not None else s_q - 1
    ts = np.unique(np.array([0, 1, first - 1] + list(range(first, s_q))))
    sub = wl.MlaInputs(q=inp.q[ts], kv=inp.kv, idx=inp.idx[ts], sink=None, sm_scale=inp.sm_scale)
    O, L = oracle_mla(sub)
    assert_cast_close(r["out"][ts], O, "e4m3", 64.0)
    assert_lse_close(r["lse"][ts], L)


def test_tail_in_graph_back_to_back():
    """100 calls captured in a CUDA graph (decode + tail combine each), replayed: no
    wait runs out and the last call's output is the oracle's."""
    s_q = 10
    inp = wl.mla_inputs(s_q, 32768, 640, seed=97, with_sink=True)
    dev = torch.device("cuda")
    q, kv, idx, sink = inp.q.to(dev), inp.kv.to(dev), inp.idx.to(dev), inp.sink.to(dev)
    plan = b.mla_decode_plan(s_q, 640, num_sms=8)
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=dev)
    out = torch.empty(s_q, 64, 512, dtype=torch.float32, device=dev)
    lse = torch.empty(s_q, 64, dtype=torch.float32, device=dev)
    st = torch.cuda.Stream()

    def call():
        b.mla_sparse_decode(plan, s_q, q, kv, inp.n_kv, idx, inp.sm_scale, sink, "f32", 1.0, out, lse, None, ws,
                            stream=st)
    with torch.cuda.stream(st):
        call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        for _ in range(50):
            call()
    with torch.cuda.stream(st):
        for _ in range(2):
            g.replay()
    torch.cuda.synchronize()
    check_status()
    O, L = oracle_mla(inp)
    assert_o_close(out.cpu().numpy(), O)
    assert_lse_close(lse.cpu().double().numpy(), L)

"""GPU parity of the sparse-MLA split-KV decode path against the fp64 oracle.

Every call goes through the C ABI (libsplitkv.so) via the ctypes binding.
Cases follow the pages' workloads (FlashMLA PR #25: h_q = 64, topk 128+512;
its test matrix s_q {1, 6, 16} x splits {2, 4, 8} x sink {off, on}, a
degenerate case with more splits than KV blocks, and the unsplit FP8 output),
plus ragged top-k, padding, out-of-range indices, the lazy-rescale path, graph
capture and the bounded-wait abort path. Tolerances: see _gpu_util.
"""
import math

import numpy as np
import pytest
import torch

import oracle.mla as om
from _gpu_util import (assert_cast_close, assert_lse_close, assert_o_close, check_status, oracle_mla,
                       run_mla, workspace_views)
from split_kv_sparse_gb300 import binding as b
from split_kv_sparse_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "the -m gpu tests need a CUDA GPU"
    b.lib()            # fails loudly if the library is missing
    check_status()


# ---- small config: s_q = 1, 4096 rows, 640 distinct uniform indices, S in {1, 4} ----------

@pytest.mark.parametrize("S", [1, 4])
def test_small_config(S):
    inp = wl.mla_inputs(1, 4096, 640, seed=0, index_mode="uniform")
    O, L = oracle_mla(inp)
    r = run_mla(inp, S)
    assert_o_close(r["out"].numpy(), O)
    assert_lse_close(r["lse"], L)


# ---- the page's test matrix on a 32768-row cache ---------------------------------------

@pytest.mark.parametrize("s_q", [1, 6, 16])
@pytest.mark.parametrize("with_sink", [False, True])
@pytest.mark.parametrize("v_mean", [0.0, 1.0])
def test_matrix(s_q, with_sink, v_mean):
    inp = wl.mla_inputs(s_q, 32768, 640, seed=10 + s_q, v_mean=v_mean, with_sink=with_sink)
    O, L = oracle_mla(inp)
    for S in (2, 4, 8):
        r = run_mla(inp, S)
        assert_o_close(r["out"].numpy(), O, what=f"O S={S}")
        assert_lse_close(r["lse"], L, what=f"LSE S={S}")


@pytest.mark.parametrize("S", [2, 3, 8, 10, 16])
def test_split_partials_match_oracle(S):
    """Each split's fp32 partial O and log2 LSE in the workspace, against the oracle's partials."""
    inp = wl.mla_inputs(3, 32768, 640, seed=21)
    O_s, L_s = om.split_partials(inp.q, inp.kv, inp.idx, inp.sm_scale, S)
    r = run_mla(inp, S, keep_workspace=True)
    for s in range(S):
        assert_o_close(r["o_acc"][s], O_s[s], what=f"partial O split {s}")
        assert_lse_close(r["lse_acc"][s], L_s[s], what=f"partial LSE split {s}")


@pytest.mark.parametrize("num_sms,D", [(152, 4), (40, 2), (20, 1)])
@pytest.mark.parametrize("S", [1, 5])
def test_dim_groups(S, num_sms, D):
    """A (token, split) job's dims spread over D CTAs (chosen by the plan from the SM
    count): partials, final O, LSE and amax as with one CTA per job."""
    inp = wl.mla_inputs(4, 32768, 640, seed=61, v_mean=1.0, with_sink=True)
    O, L = oracle_mla(inp)
    r = run_mla(inp, S, out_dtype="bf16", with_amax=True, keep_workspace=True, num_sms=num_sms)
    assert r["plan"].dim_groups == (D if S == 5 else max(d for d in (4, 2, 1) if 4 * d <= num_sms or d == 1))
    assert_cast_close(r["out"], O, "bf16")
    assert_lse_close(r["lse"], L)
    assert abs(r["amax"] - float(np.abs(O).max())) <= 2e-3 * float(np.abs(O).max())
    if S > 1:
        O_s, L_s = om.split_partials(inp.q, inp.kv, inp.idx, inp.sm_scale, S)
        for s in range(S):
            assert_o_close(r["o_acc"][s], O_s[s], what=f"partial O split {s}")
            assert_lse_close(r["lse_acc"][s], L_s[s], what=f"partial LSE split {s}")


def test_degenerate_more_splits_than_blocks():
    """s_q = 4, topk = 64 with per-token valid counts in [1, 64] (rest -1), 16 splits over 1 block."""
    inp = wl.mla_inputs(4, 32768, 64, seed=3, index_mode="padded", with_sink=True)
    O, L = oracle_mla(inp)
    r = run_mla(inp, 16, keep_workspace=True)
    assert np.all(r["o_acc"][1:] == 0) and np.all(np.isneginf(r["lse_acc"][1:]))
    O_s, L_s = om.split_partials(inp.q, inp.kv, inp.idx, inp.sm_scale, 16)
    assert_o_close(r["o_acc"][0], O_s[0])
    assert_lse_close(r["lse_acc"][0], L_s[0])
    assert_o_close(r["out"].numpy(), O)
    assert_lse_close(r["lse"], L)


@pytest.mark.parametrize("topk,s_q,S", [(1, 2, 1), (10, 3, 1), (63, 2, 2), (65, 2, 2), (200, 5, 3),
                                         (200, 5, 1), (1000, 2, 7), (2048, 1, 16), (129, 1, 1)])
def test_ragged_topk(topk, s_q, S):
    inp = wl.mla_inputs(s_q, 4096, topk, seed=topk, index_mode="uniform", with_sink=(topk % 2 == 0))
    O, L = oracle_mla(inp)
    r = run_mla(inp, S)
    assert_o_close(r["out"].numpy(), O)
    assert_lse_close(r["lse"], L)


def test_padding_out_of_range_duplicates_and_empty_token():
    inp = wl.mla_inputs(4, 4096, 256, seed=5, index_mode="uniform", with_sink=True)
    idx = inp.idx.clone()
    idx[0, :] = -1                         # nothing to attend: O = 0, LSE = -inf even with a sink
    idx[1, 10:50] = 4096 + 13              # past the end of the cache: masked
    idx[1, 50:60] = -7                     # any negative index is masked
    idx[2, 1::2] = idx[2, 0::2]            # duplicates count twice
    idx[3, 64:] = -1                       # only the first block is valid
    inp.idx = idx
    O, L = oracle_mla(inp)
    for S in (1, 2, 4):
        r = run_mla(inp, S)
        assert np.all(r["out"].numpy()[0] == 0) and np.all(np.isneginf(r["lse"][0]))
        assert_o_close(r["out"].numpy(), O)
        assert_lse_close(r["lse"], L)


def _rising_scores(s_q, topk, seed, step_natural=0.13, descending=False):
    """Scores that rise along the top-k order by ~8.3 natural units (12 log2 units)
    per 64 rows, so the running max moves past the lazy-rescale threshold at every
    block. They rise from about -166 to 0 (or fall, when descending), so the LSE
    stays small: at |LSE| ~ 240 a single fp32 ulp is already 1.5e-5, which no fp32
    kernel can hold to the 1e-5 absolute LSE tolerance."""
    rng = np.random.default_rng(seed)
    n_kv = 4096
    u = np.zeros(576, np.float32)
    u[0] = 1.0
    kv = (0.05 * rng.standard_normal((n_kv, 576))).astype(np.float32)
    idx = rng.permutation(n_kv)[: s_q * topk].reshape(s_q, topk).astype(np.int32)   # disjoint per token
    a = step_natural * (np.arange(topk, dtype=np.float32) - (topk - 1))
    if descending:
        a = a[::-1].copy()
    for t in range(s_q):
        kv[idx[t], 0] = a
    q = np.zeros((s_q, 64, 576), np.float32)
    q[:, :, 0] = 24.0 * (1.0 + np.arange(64) / 64.0)[None, :]
    q += (0.05 * rng.standard_normal(q.shape)).astype(np.float32)
    return wl.MlaInputs(q=torch.from_numpy(q).bfloat16(), kv=torch.from_numpy(kv).bfloat16(),
                        idx=torch.from_numpy(idx), sink=None, sm_scale=1.0 / 24.0)


@pytest.mark.parametrize("descending", [False, True])
@pytest.mark.parametrize("S", [1, 2, 5])
def test_lazy_rescale_path(descending, S):
    inp = _rising_scores(2, 640, seed=7, descending=descending)
    O, L = oracle_mla(inp)
    r = run_mla(inp, S)
    assert_o_close(r["out"].numpy(), O)
    assert_lse_close(r["lse"], L)


@pytest.mark.parametrize("out_dtype", ["bf16", "e4m3"])
@pytest.mark.parametrize("S", [1, 4])
@pytest.mark.parametrize("v_mean", [0.0, 1.0])
def test_output_casts_and_amax(out_dtype, S, v_mean):
    inp = wl.mla_inputs(6, 32768, 640, seed=31, v_mean=v_mean, with_sink=True)
    O, L = oracle_mla(inp)
    inv_scale = 64.0 if out_dtype == "e4m3" else 1.0
    r = run_mla(inp, S, out_dtype=out_dtype, inv_scale=inv_scale, with_amax=True)
    same = assert_cast_close(r["out"], O, out_dtype, inv_scale)
    if v_mean == 1.0:
        # FlashMLA PR #25, "Test plan": 99.6% identical FP8 codes with non-cancelling values
        assert same >= 0.99, f"only {same:.4f} of the codes equal the oracle's"
    assert_lse_close(r["lse"], L)
    amax_ref = float(np.max(np.abs(O)))
    assert abs(r["amax"] - amax_ref) <= 2e-3 * amax_ref


def test_split_equals_direct_closely():
    """The split + combine path and the direct path agree with each other (LSE to 1e-5)."""
    inp = wl.mla_inputs(16, 32768, 640, seed=44, with_sink=True)
    r1 = run_mla(inp, 1)
    for S in (2, 5, 10):
        rs = run_mla(inp, S)
        assert_o_close(rs["out"].numpy(), r1["out"].double().numpy())
        assert_lse_close(rs["lse"], r1["lse"])


def test_cuda_graph_capture_and_replay():
    inp = wl.mla_inputs(6, 32768, 640, seed=9, with_sink=True)
    dev = torch.device("cuda")
    q, kv, idx, sink = inp.q.to(dev), inp.kv.to(dev), inp.idx.to(dev), inp.sink.to(dev)
    plan = b.mla_decode_plan(16, 640)          # one plan for the whole s_q <= 16 bucket
    assert plan.num_splits > 1
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=dev)
    b.mla_workspace_init(plan, ws)
    out = torch.empty(6, 64, 512, dtype=torch.uint8, device=dev)
    lse = torch.empty(6, 64, dtype=torch.float32, device=dev)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        b.mla_sparse_decode(plan, 6, q, kv, inp.n_kv, idx, inp.sm_scale, sink, "e4m3", 64.0, out, lse, None, ws,
                            stream=s)
    torch.cuda.synchronize()
    eager = out.clone()
    eager_lse = lse.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        b.mla_sparse_decode(plan, 6, q, kv, inp.n_kv, idx, inp.sm_scale, sink, "e4m3", 64.0, out, lse, None, ws,
                            stream=s)
    out.zero_()
    lse.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    check_status()
    assert torch.equal(out, eager)
    assert torch.equal(lse, eager_lse)


def test_bounded_wait_gives_up_and_context_survives():
    check_status()
    b.mla_selftest_wait_timeout(2_000_000)     # 2 ms on a barrier nothing arrives on
    st, site = b.mla_get_status()
    assert st & b.MLA_STATUS_TIMEOUT and site == 0x5E1F
    assert b.mla_get_status() == (0, 0)        # read-and-clear
    # the context is still usable
    inp = wl.mla_inputs(1, 4096, 128, seed=1, index_mode="uniform")
    O, L = oracle_mla(inp)
    r = run_mla(inp, 2)
    assert_o_close(r["out"].numpy(), O)


def test_host_errors_on_gpu():
    inp = wl.mla_inputs(2, 4096, 640, seed=2, index_mode="uniform")
    dev = torch.device("cuda")
    q, kv, idx = inp.q.to(dev), inp.kv.to(dev), inp.idx.to(dev)
    plan = b.mla_decode_plan(2, 640, force_splits=4)
    small = torch.empty(64, dtype=torch.uint8, device=dev)
    out = torch.empty(2, 64, 512, device=dev)
    with pytest.raises(b.SplitKVError) as e:
        b.mla_sparse_decode(plan, 3, q, kv, inp.n_kv, idx, inp.sm_scale, None, "f32", 1.0, out, None, None, small)
    assert e.value.status == 1
    with pytest.raises(b.SplitKVError) as e:
        b.mla_sparse_decode(plan, 2, q[:, :, 1:], kv, inp.n_kv, idx, inp.sm_scale, None, "f32", 1.0, out, None,
                            None, small)
    assert e.value.status == 1                 # q not 16-byte aligned
    check_status()


# ---- the bench's workload at full size: every swept (s_q, splits) point, every token ---

SWEEP_N_KV = 131072
SWEEP_TOPK = 640


@pytest.fixture(scope="module")
def sweep_cache():
    """The bench's inputs: one 131072-row cache (seed 0) and, per s_q, its queries and
    128 + 512 indices (seed 1000 + s_q), with the oracle's O and LSE of every token."""
    base = wl.mla_inputs(1, SWEEP_N_KV, SWEEP_TOPK, seed=0)
    cache = {}

    def get(s_q):
        if s_q not in cache:
            inp = wl.mla_inputs(s_q, SWEEP_N_KV, SWEEP_TOPK, seed=1000 + s_q) if s_q != 1 else base
            inp = wl.MlaInputs(q=inp.q, kv=base.kv, idx=inp.idx, sink=None, sm_scale=inp.sm_scale)
            O, L = oracle_mla(inp)
            cache[s_q] = (inp, O, L)
        return cache[s_q]
    return get


@pytest.mark.parametrize("S", [1, 2, 4, 8, 16, 0, b.MLA_FORCE_BALANCED])
@pytest.mark.parametrize("s_q", [1, 6, 16, 96, 384])
def test_sweep_point_every_token(sweep_cache, s_q, S):
    """Each (s_q, num_splits) point the bench times (forced splits, the planner's choice,
    the balanced schedule where it applies), on the bench's inputs, over the device's SMs:
    every token in fp32 (row-wise 2e-3, LSE 1e-5) and as the bench's e4m3 output (every
    code within one step of the oracle's, LSE 1e-5)."""
    inp, O, L = sweep_cache(s_q)
    r = run_mla(inp, S)
    if S == b.MLA_FORCE_BALANCED and r["plan"].balanced_ctas == 0:
        pytest.skip("the balanced schedule does not apply at this s_q (the bench skips it too)")
    assert_o_close(r["out"].numpy(), O)
    assert_lse_close(r["lse"], L)
    r8 = run_mla(inp, S, out_dtype="e4m3", inv_scale=64.0)
    assert_cast_close(r8["out"], O, "e4m3", 64.0)
    assert_lse_close(r8["lse"], L)


def test_many_tokens_sampled():
    """1000 tokens: seven waves of (token) CTAs on 152 SMs, the automatic plan."""
    inp = wl.mla_inputs(1000, 131072, 640, seed=6)
    r = run_mla(inp, 0, out_dtype="bf16")
    ts = np.array([0, 151, 152, 607, 999])
    sub = wl.MlaInputs(q=inp.q[ts], kv=inp.kv, idx=inp.idx[ts], sink=None, sm_scale=inp.sm_scale)
    O, L = oracle_mla(sub)
    assert_cast_close(r["out"][ts], O, "bf16")
    assert_lse_close(r["lse"][ts], L)


def test_long_topk():
    """topk 4096 (64 blocks): many splits of several blocks each."""
    inp = wl.mla_inputs(2, 32768, 4096, seed=8, index_mode="uniform", with_sink=True)
    O, L = oracle_mla(inp)
    for S in (0, 7, 64):
        r = run_mla(inp, S)
        assert_o_close(r["out"].numpy(), O, what=f"O S={S}")
        assert_lse_close(r["lse"], L, what=f"LSE S={S}")


@pytest.mark.parametrize("S", [1, 2])
def test_dim_groups_on_long_top_k(S):
    """A job's dims spread over four CTAs (the plan for two tokens on the device's SMs) on
    topk 4096: 64 or 32 steps per CTA, so any drift in how a CTA releases ring
    chunks to its loaders would show as a wrong row, a wrong result or a timeout."""
    inp = wl.mla_inputs(2, 32768, 4096, seed=88, index_mode="uniform", with_sink=True)
    O, L = oracle_mla(inp)
    r = run_mla(inp, S)
    assert r["plan"].dim_groups == 4
    assert_o_close(r["out"].numpy(), O)
    assert_lse_close(r["lse"], L)


@pytest.mark.parametrize("s_q,S", [(1, 0), (6, 0), (96, 0), (16, b.MLA_FORCE_BALANCED), (2, 1)])
def test_many_calls_back_to_back(s_q, S):
    """200 consecutive decode calls in CUDA graphs, as the bench runs them: no wait
    may run out, and the last call's output is the oracle's."""
    inp = wl.mla_inputs(s_q, 32768, 640, seed=900 + s_q, with_sink=True)
    dev = torch.device("cuda")
    q, kv, idx, sink = inp.q.to(dev), inp.kv.to(dev), inp.idx.to(dev), inp.sink.to(dev)
    plan = b.mla_decode_plan(s_q, 640, force_splits=S)
    ws = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device=dev)
    if plan.workspace_bytes:
        b.mla_workspace_init(plan, ws)
    out = torch.empty(s_q, 64, 512, dtype=torch.float32, device=dev)
    lse = torch.empty(s_q, 64, dtype=torch.float32, device=dev)
    st = torch.cuda.Stream()

    def call():
        b.mla_sparse_decode(plan, s_q, q, kv, inp.n_kv, idx, inp.sm_scale, sink, "f32", 1.0, out, lse, None,
                            ws if plan.workspace_bytes else None, stream=st)
    with torch.cuda.stream(st):
        call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        for _ in range(50):
            call()
    with torch.cuda.stream(st):
        for _ in range(4):
            g.replay()
    torch.cuda.synchronize()
    check_status()
    O, L = oracle_mla(inp)
    assert_o_close(out.cpu().numpy(), O)
    assert_lse_close(lse.cpu().double().numpy(), L)


def test_cache_past_two_gigabytes():
    """A 2.1M-row cache (2.4 GB, row offsets past 2^31 bytes), made of copies of a
    32768-row seeded cache; the indices reach the last rows."""
    base = wl.mla_inputs(3, 32768, 640, seed=12, index_mode="uniform")
    n_kv = 2_100_000
    dev = torch.device("cuda")
    kv = base.kv.to(dev).repeat(-(-n_kv // 32768), 1)[:n_kv].contiguous()
    g = torch.Generator().manual_seed(12)
    idx = torch.randint(n_kv - 300_000, n_kv, (3, 640), generator=g, dtype=torch.int64)
    idx[:, :64] = torch.arange(n_kv - 64, n_kv)          # the very last rows
    idx = idx.to(torch.int32)
    sub = wl.MlaInputs(q=base.q, kv=base.kv, idx=(idx.long() % 32768).to(torch.int32), sink=None,
                       sm_scale=base.sm_scale)
    O, L = oracle_mla(sub)
    for S in (1, 4):
        plan = b.mla_decode_plan(3, 640, force_splits=S)
        ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=dev) if plan.workspace_bytes else None
        out = torch.empty(3, 64, 512, dtype=torch.float32, device=dev)
        lse = torch.empty(3, 64, dtype=torch.float32, device=dev)
        b.mla_sparse_decode(plan, 3, base.q.to(dev), kv, n_kv, idx.to(dev), base.sm_scale, None, "f32", 1.0, out,
                            lse, None, ws)
        torch.cuda.synchronize()
        check_status()
        assert_o_close(out.cpu().numpy(), O, what=f"O S={S}")
        assert_lse_close(lse.cpu().double().numpy(), L, what=f"LSE S={S}")
    del kv
    torch.cuda.empty_cache()


# ---- balanced schedule: range boundaries cutting tokens anywhere ----------------------

@pytest.mark.parametrize("s_q,topk,num_sms", [
    (2, 640, 5),      # 20 blocks over 5 CTAs of 4: each token in 3 pieces
    (3, 640, 4),      # 30 blocks over 4 CTAs (8, 8, 7, 7): CTAs holding pieces of two tokens
    (5, 640, 2),      # 50 blocks over 2 CTAs of 25: whole tokens beside the pieces of a cut one
    (7, 200, 5),      # ragged top-k (4 blocks, the last of 8 rows), 28 blocks over 5 CTAs
    (4, 640, 3),      # 40 blocks over 3 CTAs (14, 13, 13)
])
@pytest.mark.parametrize("with_sink", [False, True])
def test_balanced_schedule_matches_oracle(s_q, topk, num_sms, with_sink):
    inp = wl.mla_inputs(s_q, 32768, topk, seed=300 + s_q * 7 + num_sms, with_sink=with_sink,
                        index_mode="window" if topk >= 128 else "uniform")
    O, L = oracle_mla(inp)
    r = run_mla(inp, b.MLA_FORCE_BALANCED, num_sms=num_sms)
    assert r["plan"].balanced_ctas > 0
    assert_o_close(r["out"].numpy(), O)
    assert_lse_close(r["lse"], L)


@pytest.mark.parametrize("out_dtype", ["bf16", "e4m3"])
def test_balanced_schedule_casts_and_amax(out_dtype):
    """Whole tokens are cast by the decode kernel and cut tokens by the combine;
    the amax is the max over both."""
    inp = wl.mla_inputs(5, 32768, 640, seed=41, v_mean=1.0, with_sink=True)
    O, L = oracle_mla(inp)
    r = run_mla(inp, b.MLA_FORCE_BALANCED, out_dtype=out_dtype, inv_scale=64.0, with_amax=True,
                num_sms=4)   # 50 over 4
    assert_cast_close(r["out"], O, out_dtype, 64.0)
    assert_lse_close(r["lse"], L)
    assert abs(r["amax"] - float(np.abs(O).max())) <= 2e-3 * float(np.abs(O).max())


def test_balanced_schedule_padding_and_empty_pieces():
    """Padded and out-of-range indices; a piece whose rows are all masked is an
    empty partial (LSE = -inf) and drops out of the combine; a token with no valid
    row at all is O = 0, LSE = -inf."""
    inp = wl.mla_inputs(4, 32768, 640, seed=43)
    idx = inp.idx.clone()
    idx[1, 0:256] = -1             # token 1's first piece (blocks 0-3, in CTA 0) holds no valid row
    idx[3, :] = -1                 # token 3 (whole, in CTA 2): nothing valid
    idx[2, 100:110] = 40000        # out of range: masked
    inp = wl.MlaInputs(q=inp.q, kv=inp.kv, idx=idx, sink=None, sm_scale=inp.sm_scale)
    O, L = oracle_mla(inp)
    r = run_mla(inp, b.MLA_FORCE_BALANCED, num_sms=3)       # 40 blocks over 3 CTAs (14, 13, 13)
    assert r["plan"].balanced_ctas > 0
    assert_o_close(r["out"].numpy(), O)
    assert_lse_close(r["lse"], L)


def test_balanced_schedule_repeated_calls():
    """Two calls in a row on one workspace that starts out filled with garbage (no
    clearing): every partial slot a call reads was written by the same call, so both
    calls give the same, correct result."""
    inp = wl.mla_inputs(3, 32768, 640, seed=47, with_sink=True)
    O, L = oracle_mla(inp)
    dev = torch.device("cuda")
    plan = b.mla_decode_plan(3, 640, num_sms=4, force_splits=b.MLA_FORCE_BALANCED)
    assert plan.balanced_ctas > 0
    ws = torch.full((plan.workspace_bytes,), 0xA5, dtype=torch.uint8, device=dev)
    outs = []
    for _ in range(2):
        out = torch.empty(3, 64, 512, dtype=torch.float32, device=dev)
        lse = torch.empty(3, 64, dtype=torch.float32, device=dev)
        b.mla_sparse_decode(plan, 3, inp.q.to(dev), inp.kv.to(dev), inp.n_kv, inp.idx.to(dev), inp.sm_scale,
                            inp.sink.to(dev), "f32", 1.0, out, lse, None, ws)
        torch.cuda.synchronize()
        check_status()
        outs.append((out.cpu(), lse.cpu()))
    for out, lse in outs:
        assert_o_close(out.numpy(), O)
        assert_lse_close(lse.double().numpy(), L)
    assert torch.equal(outs[0][0], outs[1][0])


@pytest.mark.parametrize("s_q,S", [(6, 0), (96, 0), (16, b.MLA_FORCE_BALANCED)])
def test_host_buffer_call(s_q, S):
    """mla_sparse_decode_host: queries and indices from pinned host memory, FP8 output and LSE back to
    host memory, all on one stream; the same bytes as the device-buffer call, and the oracle's values."""
    inp = wl.mla_inputs(s_q, 32768, 640, seed=77, with_sink=True)
    dev = torch.device("cuda")
    kv, sink = inp.kv.to(dev), inp.sink.to(dev)
    plan = b.mla_decode_plan(s_q, 640, force_splits=S)
    ws = torch.empty(max(plan.workspace_bytes, 1), dtype=torch.uint8, device=dev)
    if plan.workspace_bytes:
        b.mla_workspace_init(plan, ws)
    q_h, idx_h = inp.q.pin_memory(), inp.idx.pin_memory()
    q_d, idx_d = torch.empty_like(inp.q, device=dev), torch.empty_like(inp.idx, device=dev)
    out_d = torch.empty(s_q, 64, 512, dtype=torch.uint8, device=dev)
    out_h = torch.zeros(s_q, 64, 512, dtype=torch.uint8).pin_memory()
    lse_d = torch.empty(s_q, 64, dtype=torch.float32, device=dev)
    lse_h = torch.zeros(s_q, 64, dtype=torch.float32).pin_memory()
    st = torch.cuda.Stream()
    b.mla_sparse_decode_host(plan, s_q, q_h, q_d, kv, inp.n_kv, idx_h, idx_d, inp.sm_scale, sink, "e4m3", 64.0,
                             out_d, out_h, lse_d, lse_h, None, ws if plan.workspace_bytes else None, stream=st)
    st.synchronize()
    check_status()
    r = run_mla(inp, S, out_dtype="e4m3", inv_scale=64.0)
    assert torch.equal(out_h, r["out"])
    assert np.array_equal(lse_h.double().numpy(), r["lse"])
    ts = np.array([0, s_q - 1])
    sub = wl.MlaInputs(q=inp.q[ts], kv=inp.kv, idx=inp.idx[ts], sink=inp.sink, sm_scale=inp.sm_scale)
    O, L = oracle_mla(sub)
    assert_cast_close(out_h[ts], O, "e4m3", 64.0)
    assert_lse_close(lse_h[ts].double().numpy(), L)


def _decode_status(inp, S=0):
    """One decode through mla_sparse_decode; returns (O, LSE, status bits) without asserting the status."""
    dev = torch.device("cuda")
    plan = b.mla_decode_plan(inp.s_q, inp.topk, force_splits=S)
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=dev) if plan.workspace_bytes else None
    out = torch.empty(inp.s_q, 64, 512, dtype=torch.float32, device=dev)
    lse = torch.empty(inp.s_q, 64, dtype=torch.float32, device=dev)
    b.mla_sparse_decode(plan, inp.s_q, inp.q.to(dev), inp.kv.to(dev), inp.n_kv, inp.idx.to(dev), inp.sm_scale, None,
                        "f32", 1.0, out, lse, None, ws)
    st, _ = b.mla_get_status()
    return out.cpu().numpy(), lse.cpu().double().numpy(), st


@pytest.mark.parametrize("S", [0, 1])
def test_index_checks_report_corrupt_indices(S):
    """With index checks on, an index outside {-1} and [0, n_kv) sets MLA_STATUS_BAD_INDEX;
    -1 padding alone sets nothing; the row is masked either way (the oracle's result);
    with checks off nothing is reported."""
    inp = wl.mla_inputs(4, 32768, 640, seed=131)
    pad = inp.idx.clone()
    pad[0, 5] = -1
    pad[1, 600:640] = -1
    bad = pad.clone()
    bad[2, 10] = inp.n_kv          # one past the cache
    bad[3, 300] = -7               # negative, not the padding value
    pad_in = wl.MlaInputs(q=inp.q, kv=inp.kv, idx=pad, sink=None, sm_scale=inp.sm_scale)
    bad_in = wl.MlaInputs(q=inp.q, kv=inp.kv, idx=bad, sink=None, sm_scale=inp.sm_scale)
    O_pad, L_pad = oracle_mla(pad_in)
    O_bad, L_bad = oracle_mla(bad_in)
    b.mla_set_index_checks(True)
    try:
        o, l, st = _decode_status(pad_in, S)
        assert st == 0
        assert_o_close(o, O_pad)
        o, l, st = _decode_status(bad_in, S)
        assert st == b.MLA_STATUS_BAD_INDEX
        assert_o_close(o, O_bad)
        assert_lse_close(l, L_bad)
    finally:
        b.mla_set_index_checks(False)
    o, l, st = _decode_status(bad_in, S)
    assert st == 0
    assert_o_close(o, O_bad)

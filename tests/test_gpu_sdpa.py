"""GPU parity of the dense split-KV FP8 SDPA decode path (cuDNN-frontend PR #768
form) against the fp64 oracle, through the C ABI.

Cases: the dense workload (batch 8, 32 query / 8 KV heads, d = 128, 1-16 new
tokens per sequence, causal KV lengths in [1024, 16384], per-tensor e4m3
Q/K/V) at several split counts including the planner's, small ragged
batches, empty chunks past the end, GQA group sizes 1/4/16, every output
cast, the combine's amax, and a sequence with more rows than a job holds.
Tolerances as in _gpu_util (fp32 O row-wise 2e-3, LSE 1e-5, casts compared
after the same cast, amax 2e-3 relative).
"""
import numpy as np
import pytest
import torch

import oracle.sdpa as osd
from _gpu_util import BF16_FLOOR_DENSE, TORCH_OUT, assert_cast_close, assert_lse_close, assert_o_close, check_status
from split_kv_sparse_gb300 import binding as b
from split_kv_sparse_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "the -m gpu tests need a CUDA GPU"
    b.lib()
    check_status()


def run_sdpa(inp, S, out_dtype="f32", inv_scale=1.0, with_amax=True, keep_workspace=False, max_q=None):
    dev = torch.device("cuda")
    total_q = int(inp.cu_seqlens_q[-1])
    total_kv = int(inp.cu_seqlens_kv[-1])
    sq = (inp.cu_seqlens_q[1:] - inp.cu_seqlens_q[:-1])
    skv = (inp.cu_seqlens_kv[1:] - inp.cu_seqlens_kv[:-1])
    plan = b.sdpa_fp8_decode_plan(inp.batch, inp.h_q, inp.h_kv, inp.d, max_q or int(sq.max()), total_q,
                                  int(skv.max()), force_splits=S)
    q, k, v = inp.q.to(dev), inp.k.to(dev), inp.v.to(dev)
    cq, ck = inp.cu_seqlens_q.to(dev), inp.cu_seqlens_kv.to(dev)
    ds = [torch.tensor([x], dtype=torch.float32, device=dev) for x in (inp.descale_q, inp.descale_k, inp.descale_v)]
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=dev) if plan.workspace_bytes else None
    out = torch.empty(total_q, inp.h_q, inp.d, dtype=TORCH_OUT[out_dtype], device=dev)
    lse = torch.empty(total_q, inp.h_q, dtype=torch.float32, device=dev)
    amax = torch.empty(1, dtype=torch.float32, device=dev) if with_amax else None
    b.sdpa_fp8_decode(plan, total_q, total_kv, q, k, v, cq, ck, ds[0], ds[1], ds[2], inp.sm_scale, out_dtype,
                      inv_scale, out, lse, amax, ws)
    torch.cuda.synchronize()
    check_status()
    r = {"out": out.cpu(), "lse": lse.cpu().double().numpy(), "plan": plan}
    if with_amax:
        r["amax"] = float(amax.cpu()[0])
    if keep_workspace and ws is not None:
        Sn = plan.num_splits
        r["o_acc"] = ws[: Sn * total_q * inp.h_q * 128 * 4].view(torch.float32).view(Sn, total_q, inp.h_q, 128) \
            .cpu().double().numpy()
        off = plan.lse_acc_offset
        r["lse_acc"] = ws[off: off + Sn * total_q * inp.h_q * 4].view(torch.float32).view(Sn, total_q, inp.h_q) \
            .cpu().double().numpy()
    return r


def _check(inp, r, O, L):
    assert_o_close(r["out"].numpy(), O)
    assert_lse_close(r["lse"], L)
    amax_ref = float(np.max(np.abs(O)))
    assert abs(r["amax"] - amax_ref) <= 2e-3 * amax_ref


@pytest.mark.parametrize("S", [1, 2, 3, 5])
def test_small_ragged_batch(S):
    inp = wl.sdpa_inputs(3, 8, 2, 128, q_per_seq=(1, 5), kv_len=(40, 700), seed=1)
    O, L = osd.attention(inp)
    _check(inp, run_sdpa(inp, S), O, L)


def test_split_partials_and_empty_chunks():
    inp = wl.sdpa_inputs(4, 8, 2, 128, q_per_seq=(1, 4), kv_len=(100, 300), seed=2)   # <= 3 tiles per sequence
    S = 5
    O_s, L_s = osd.split_partials(inp, S)
    r = run_sdpa(inp, S, keep_workspace=True)
    for s in range(S):
        assert_o_close(r["o_acc"][s], O_s[s], what=f"partial O split {s}")
        assert_lse_close(r["lse_acc"][s], L_s[s], what=f"partial LSE split {s}")


@pytest.mark.parametrize("h_q,h_kv,q_per_seq", [(8, 8, (1, 16)), (16, 1, (1, 4)), (32, 8, (1, 16))])
def test_group_sizes(h_q, h_kv, q_per_seq):
    inp = wl.sdpa_inputs(3, h_q, h_kv, 128, q_per_seq=q_per_seq, kv_len=(129, 1500), seed=h_q)
    O, L = osd.attention(inp)
    for S in (1, 4):
        _check(inp, run_sdpa(inp, S), O, L)


def test_adaptive_splits_on_a_ragged_batch():
    """The planner's per-sequence split counts: a long sequence beside short ones.
    Final O / LSE as the oracle; the split slots a sequence does not use hold
    LSE = -inf."""
    inp = wl.sdpa_inputs(4, 8, 2, 128, q_per_seq=(1, 4), kv_len=(100, 20000), seed=9)
    O, L = osd.attention(inp)
    r = run_sdpa(inp, 0, keep_workspace=True)
    assert r["plan"].adaptive_splits == 1
    _check(inp, r, O, L)
    skv = (inp.cu_seqlens_kv[1:] - inp.cu_seqlens_kv[:-1]).tolist()
    cq = inp.cu_seqlens_q.tolist()
    # some sequence uses fewer splits than the bound: its last slot is -inf, its first is not
    unused = [b for b in range(4) if np.all(np.isneginf(r["lse_acc"][-1, cq[b]:cq[b + 1]]))]
    assert unused, "every sequence used every split slot"
    for b in unused:
        assert np.all(np.isfinite(r["lse_acc"][0, cq[b]:cq[b + 1]]))
    assert max(skv) > 8 * 128


def test_single_key_sequences():
    inp = wl.sdpa_inputs(4, 8, 2, 128, q_per_seq=(1, 1), kv_len=(1, 1), seed=3)
    O, L = osd.attention(inp)
    for S in (1, 2):
        _check(inp, run_sdpa(inp, S), O, L)


@pytest.fixture(scope="module")
def full_case():
    inp = wl.sdpa_inputs(8, 32, 8, 128, seed=0)
    O, L = osd.attention(inp)
    return inp, O, L


@pytest.mark.parametrize("S", [0, 1, 2, 4, 16])
def test_full_workload(full_case, S):
    inp, O, L = full_case
    _check(inp, run_sdpa(inp, S, max_q=16), O, L)


@pytest.mark.parametrize("out_dtype", ["bf16", "e4m3"])
@pytest.mark.parametrize("S", [1, 3])
def test_output_casts(full_case, out_dtype, S):
    inp, O, L = full_case
    inv_scale = 64.0 if out_dtype == "e4m3" else 1.0
    r = run_sdpa(inp, S, out_dtype=out_dtype, inv_scale=inv_scale, max_q=16)
    assert_cast_close(r["out"], O, out_dtype, inv_scale, bf16_floor=BF16_FLOOR_DENSE)
    assert_lse_close(r["lse"], L)


def test_too_many_rows_is_reported_not_computed():
    """32 query heads per KV head x 3 tokens = 96 rows > 64: the job refuses and says so."""
    inp = wl.sdpa_inputs(1, 32, 1, 128, q_per_seq=(3, 3), kv_len=(200, 200), seed=4)
    dev = torch.device("cuda")
    out = torch.full((3, 32, 128), 7.0, device=dev)
    b.sdpa_fp8_decode_direct(1, 32, 1, 128, 3, 200, inp.q.to(dev), inp.k.to(dev), inp.v.to(dev),
                             inp.cu_seqlens_q.to(dev), inp.cu_seqlens_kv.to(dev), None, None, None, inp.sm_scale,
                             "f32", 1.0, out)
    st, _ = b.mla_get_status()
    assert st & b.MLA_STATUS_BAD_SHAPE
    assert torch.all(out == 7.0)


@pytest.mark.parametrize("S", [0, 1, 3])
def test_empty_sequences(S):
    """A batch holding a sequence with no new tokens and no keys, and one with keys but
    no new tokens: their jobs have no rows (nothing written), the other sequences are
    the oracle's, with the planner's per-sequence splits, unsplit and forced splits."""
    import dataclasses
    base = wl.sdpa_inputs(5, 8, 2, 128, q_per_seq=(1, 3), kv_len=(200, 900), seed=23)
    cq = base.cu_seqlens_q.tolist()
    ck = base.cu_seqlens_kv.tolist()
    # sequence 1: drop its queries and its keys; sequence 3: drop its queries only
    keep_q = [i for i in range(cq[-1]) if not (cq[1] <= i < cq[2] or cq[3] <= i < cq[4])]
    keep_k = [i for i in range(ck[-1]) if not (ck[1] <= i < ck[2])]
    sq = [cq[b + 1] - cq[b] for b in range(5)]
    sk = [ck[b + 1] - ck[b] for b in range(5)]
    sq[1] = sq[3] = 0
    sk[1] = 0
    new_cq = torch.tensor([0] + list(np.cumsum(sq)), dtype=torch.int32)
    new_ck = torch.tensor([0] + list(np.cumsum(sk)), dtype=torch.int32)
    inp = dataclasses.replace(base, q=base.q[keep_q], k=base.k[keep_k], v=base.v[keep_k],
                              cu_seqlens_q=new_cq, cu_seqlens_kv=new_ck)
    assert int(new_cq[-1]) == len(keep_q) and int(new_ck[-1]) == len(keep_k)
    O, L = osd.attention(inp)
    _check(inp, run_sdpa(inp, S, max_q=3), O, L)

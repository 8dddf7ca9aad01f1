"""Host-side tests of the C ABI (no GPU needed).

* libsplitkv.so builds for sm_103a, loads without a GPU, and exports every
  function include/mla_split.h declares;
* the planner: workspace formula against the sizes printed in FlashMLA PR #25
  ("Measured"), determinism (a pure function of its arguments, so a CUDA graph
  bucket sees one split count), the automatic rule, forcing, and error codes;
* argument checks that run before any device work return their codes.
"""
import ctypes
import os
import re

import pytest

import oracle.mla as om
from split_kv_sparse_gb300 import binding as b
from split_kv_sparse_gb300 import build as bld

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built_library():
    if not os.path.exists(b.LIB_PATH):
        bld.build()
    return b.lib()


def _declared_functions():
    names = []
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            names += re.findall(r"^MLA_API\s+[\w\s\*]+?\b(\w+)\(", src, flags=re.M)
    return names


def test_library_exports_every_declared_function():
    declared = _declared_functions()
    assert len(declared) >= 14
    assert sorted(declared) == sorted(b.EXPORTS)
    L = ctypes.CDLL(b.LIB_PATH)
    for name in declared:
        assert hasattr(L, name), name


def test_abi_version_matches_header():
    src = open(os.path.join(ROOT, "include", "mla_split.h")).read()
    v = int(re.search(r"#define MLA_ABI_VERSION (\d+)", src).group(1))
    assert b.mla_abi_version() == v


def test_status_strings():
    for code in range(6):
        assert b.status_string(code) != "unknown status"
    assert b.status_string(99) == "unknown status"


@pytest.mark.parametrize("S,s_q", [(8, 1), (8, 16)])
def test_workspace_matches_page(S, s_q):
    p = b.mla_decode_plan(s_q, 640, num_sms=152, force_splits=S)
    assert p.o_acc_bytes == om.workspace_bytes(S, s_q) == S * s_q * 64 * 512 * 4
    assert p.lse_acc_offset % 256 == 0 and p.lse_acc_offset >= p.o_acc_bytes
    assert p.lse_acc_bytes == S * s_q * 64 * 4
    assert p.workspace_bytes >= p.lse_acc_offset + p.lse_acc_bytes and p.workspace_bytes % 256 == 0


def balanced_slots(s_q_max, nb, sms):
    """The most pieces one token is cut into by the balanced schedule over every s_q up
    to s_q_max where it applies (the blocks of all tokens cut into P near-equal ranges,
    the first U mod P one block longer), restated from the header."""
    most = 1
    for s in range(1, s_q_max + 1):
        U = s * nb
        per = -(-U // sms)
        if per < 2:
            continue
        if per > nb:
            return max(most, 2)
        P = -(-U // per)
        base, rem = divmod(U, P)
        big = rem * (base + 1)
        cta = lambda u: u // (base + 1) if u < big else rem + (u - big) // base
        for t in range(s):
            most = max(most, cta((t + 1) * nb - 1) - cta(t * nb) + 1)
    return most


def test_plan_is_deterministic_and_follows_rule():
    for sms in [148, 152, 160, 188]:
        for s_q in [1, 2, 4, 6, 8, 16, 32, 96, 384]:
            for topk in [64, 128, 640, 2048]:
                p1 = b.mla_decode_plan(s_q, topk, num_sms=sms)
                p2 = b.mla_decode_plan(s_q, topk, num_sms=sms)
                assert bytes(p1) == bytes(p2)
                nblk = -(-topk // 64)
                S = p1.num_splits
                assert 1 <= S <= nblk
                assert s_q * S <= max(sms, s_q)
                smax = max(1, min(sms // s_q, nblk, 64))
                eff = lambda c: max(2, -(-nblk // c))   # one- and two-block splits count alike
                best = eff(smax)
                S2 = next(c for c in range(1, smax + 1) if eff(c) == best)
                # ... unless every one-block split still gets 4 dim groups
                if S2 > 1 and nblk <= smax and s_q * nblk * 4 <= sms:
                    assert S == nblk
                else:
                    assert S == S2
                # uniform workspace (0 for one split), and with the automatic
                # choice also the balanced schedule's partial slots
                ru = lambda x: -(-x // 256) * 256
                uni = 0 if S == 1 else ru(ru(S * s_q * 64 * 512 * 4) + S * s_q * 64 * 4)
                per = -(-(s_q * nblk) // sms)
                applies = per >= 2
                enabled = False          # the balanced schedule only on request
                C = 0
                # one partial slot per piece of the most cut token, split layout
                slots = balanced_slots(s_q, nblk, sms)
                partials = ru(ru(slots * s_q * 64 * 512 * 4) + slots * s_q * 64 * 4)
                assert p1.balanced_ctas == C
                # CTAs per (token, split) job: 4, 2 or 1, whatever still fits the SMs
                assert p1.dim_groups == next(d for d in (4, 2, 1) if s_q * S * d <= sms or d == 1)
                # a one-split grid of more than one wave may cut its last wave's
                # tokens: up to num_sms (split, token) partial slots
                tail = sms if (S == 1 and s_q > sms and nblk >= 2) else 0
                assert p1.tail_ctas == tail
                tail_ws = ru(ru(tail * 64 * 512 * 4) + tail * 64 * 4) if tail else 0
                assert p1.workspace_bytes == max(max(uni, partials) if enabled else uni, tail_ws)
                pf = b.mla_decode_plan(s_q, topk, num_sms=sms, force_splits=S)
                assert pf.balanced_ctas == 0 and pf.tail_ctas == 0 and (pf.workspace_bytes == 0) == (S == 1)
                pb = b.mla_decode_plan(s_q, topk, num_sms=sms, force_splits=b.MLA_FORCE_BALANCED)
                assert pb.num_splits == S
                assert pb.balanced_ctas == (min(sms, s_q * nblk) if applies else 0)


def test_plan_examples():
    assert b.mla_decode_plan(1, 640, num_sms=152).num_splits == 10     # 1 block each (4 dim groups fit)
    assert b.mla_decode_plan(1, 640, num_sms=152).dim_groups == 4      # 40 CTAs
    assert b.mla_decode_plan(3, 640, num_sms=152).num_splits == 10     # 120 CTAs
    assert b.mla_decode_plan(4, 640, num_sms=152).num_splits == 5      # 160 would not fit: 2 blocks each
    assert b.mla_decode_plan(6, 640, num_sms=152).dim_groups == 4      # 5 splits, 120 CTAs
    assert b.mla_decode_plan(10, 640, num_sms=152).dim_groups == 2     # 5 splits, 100 CTAs
    assert b.mla_decode_plan(16, 640, num_sms=152).dim_groups == 1     # 5 splits, 80 CTAs
    assert b.mla_decode_plan(1, 640, num_sms=10).dim_groups == 2       # 5 splits
    assert b.mla_decode_plan(1, 640, num_sms=5).dim_groups == 1
    assert b.mla_decode_plan(1, 128, num_sms=152).num_splits == 1     # 2 blocks: no split
    assert b.mla_decode_plan(16, 640, num_sms=152).num_splits == 5
    assert b.mla_decode_plan(96, 640, num_sms=152).num_splits == 1
    assert b.mla_decode_plan(1, 640, num_sms=152, max_splits=4).num_splits == 4
    assert b.mla_decode_plan(1, 640, num_sms=152, max_splits=8).num_splits == 5
    p = b.mla_decode_plan(4, 64, num_sms=152, force_splits=16)   # more splits than blocks
    assert p.num_splits == 16 and p.num_blocks == 1


@pytest.mark.parametrize("kw,code", [
    (dict(h_q=32), 2), (dict(d_qk=512), 2), (dict(d_v=576), 2),
    (dict(force_splits=65), 1), (dict(force_splits=-2), 1), (dict(max_splits=-1), 1), (dict(num_sms=-1), 1),
])
def test_plan_errors(kw, code):
    with pytest.raises(b.SplitKVError) as e:
        b.mla_decode_plan(1, 640, **({"num_sms": 152} | kw))
    assert e.value.status == code


def test_plan_rejects_bad_sizes():
    for s_q, topk in [(0, 640), (1, 0), (-3, 640)]:
        with pytest.raises(b.SplitKVError) as e:
            b.mla_decode_plan(s_q, topk, num_sms=152)
        assert e.value.status == 1


def test_split_call_argument_checks_before_device_work():
    plan = b.mla_decode_plan(4, 640, num_sms=152, force_splits=4)
    fake = 1 << 20   # never dereferenced: every case below fails its host check first
    cases = [
        dict(s_q=5),                      # s_q > s_q_max
        dict(s_q=0),
        dict(q=None), dict(kv=None), dict(idx=None),
        dict(q=fake + 8),                 # q not 16-byte aligned
        dict(n_kv=0),
        dict(sm_scale=float("nan")),
    ]
    for c in cases:
        args = dict(s_q=2, q=fake, kv=fake, n_kv=100, idx=fake, sm_scale=0.1, workspace=fake) | c
        with pytest.raises(b.SplitKVError) as e:
            b.mla_sparse_decode_split(plan, args["s_q"], args["q"], args["kv"], args["n_kv"], args["idx"],
                                      args["sm_scale"], args["workspace"], stream=0)
        assert e.value.status == 1, c
    with pytest.raises(b.SplitKVError) as e:   # workspace missing
        b.mla_sparse_decode_split(plan, 2, fake, fake, 100, fake, 0.1, None, stream=0)
    assert e.value.status == 3
    plan1 = b.mla_decode_plan(4, 640, num_sms=152, force_splits=1)
    with pytest.raises(b.SplitKVError) as e:   # the split call needs S > 1
        b.mla_sparse_decode_split(plan1, 2, fake, fake, 100, fake, 0.1, fake, stream=0)
    assert e.value.status == 1


def test_host_buffer_call_argument_checks_before_device_work():
    """mla_sparse_decode_host rejects a missing buffer, a lone LSE pointer or a bad output type
    before it queues a copy."""
    plan = b.mla_decode_plan(4, 640, num_sms=152, force_splits=1)
    fake = 1 << 20   # never dereferenced
    full = dict(q_host=fake, q_dev=fake, idx_host=fake, idx_dev=fake, out_dev=fake, out_host=fake,
                lse_dev=None, lse_host=None, out_dtype="e4m3")
    cases = [dict(q_host=None), dict(q_dev=None), dict(idx_host=None), dict(idx_dev=None), dict(out_dev=None),
             dict(out_host=None), dict(lse_dev=fake), dict(lse_host=fake), dict(out_dtype=7)]
    for c in cases:
        a = full | c
        with pytest.raises(b.SplitKVError) as e:
            b.mla_sparse_decode_host(plan, 2, a["q_host"], a["q_dev"], fake, 100, a["idx_host"], a["idx_dev"],
                                     0.1, None, a["out_dtype"], 64.0, a["out_dev"], a["out_host"],
                                     a["lse_dev"], a["lse_host"], stream=0)
        assert e.value.status == 1, c
    with pytest.raises(b.SplitKVError) as e:   # s_q < 1
        b.mla_sparse_decode_host(plan, 0, fake, fake, fake, 100, fake, fake, 0.1, None, "e4m3", 64.0, fake, fake,
                                 stream=0)
    assert e.value.status == 1


def test_combine_argument_checks():
    plan = b.mla_decode_plan(4, 640, num_sms=152, force_splits=4)
    fake = 1 << 20
    with pytest.raises(b.SplitKVError) as e:
        b.mla_split_combine(plan, 2, fake, None, 7, 1.0, fake, stream=0)      # bad dtype
    assert e.value.status == 1
    with pytest.raises(b.SplitKVError) as e:
        b.mla_split_combine(plan, 2, fake, None, "e4m3", float("inf"), fake, stream=0)
    assert e.value.status == 1
    with pytest.raises(b.SplitKVError) as e:
        b.mla_split_combine(plan, 2, fake + 64, None, "f32", 1.0, fake, stream=0)   # workspace alignment
    assert e.value.status == 3


def test_no_device_is_reported_not_crashed():
    """Without a GPU, a call that passes its host checks reports MLA_ERR_NO_DEVICE."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    plan = b.mla_decode_plan(2, 640, num_sms=152, force_splits=2)
    fake = 1 << 20
    with pytest.raises(b.SplitKVError) as e:
        b.mla_sparse_decode_split(plan, 2, fake, fake, 100, fake, 0.1, fake, stream=0)
    assert e.value.status == 5


def test_dense_plan():
    p = b.sdpa_fp8_decode_plan(8, 32, 8, 128, 16, 128, 16384, num_sms=152)
    assert p.num_splits == 16 and p.adaptive_splits == 1   # per-sequence counts, at most 16
    pf = b.sdpa_fp8_decode_plan(8, 32, 8, 128, 16, 128, 16384, num_sms=152, force_splits=4)
    assert pf.num_splits == 4 and pf.adaptive_splits == 0
    p1 = b.sdpa_fp8_decode_plan(8, 32, 8, 128, 16, 128, 100, num_sms=152)   # one tile: no split
    assert p1.num_splits == 1 and p1.adaptive_splits == 0 and p1.workspace_bytes == 0
    assert p.o_acc_bytes == (p.num_splits * 128 * 32 * 128 * 4 if p.num_splits > 1 else 0)
    with pytest.raises(b.SplitKVError) as e:
        b.sdpa_fp8_decode_plan(8, 32, 8, 64, 16, 128, 16384, num_sms=152)
    assert e.value.status == 2
    with pytest.raises(b.SplitKVError) as e:   # 4 heads per group x 17 tokens > 64 rows per job
        b.sdpa_fp8_decode_plan(8, 32, 8, 128, 17, 128, 16384, num_sms=152)
    assert e.value.status == 2


def test_build_targets_sm103a_only():
    assert bld.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def _bal_begin(p, U, P):
    base, rem = divmod(U, P)
    return p * base + min(p, rem)


def test_balanced_schedule_covers_every_block_once():
    """The balanced one-shot schedule, restated on the host: P contiguous ranges
    of the token-major block list, near-equal; each range's jobs one per token it
    touches; every (token, block) lands in exactly one job, a token held by one
    CTA is whole, and only a CTA's first and last job can be pieces (its two
    partial slots)."""
    for sms in [148, 152]:
        for s_q in [1, 3, 6, 16, 95, 96, 97, 384]:
            for nb in [1, 2, 10, 32]:
                U = s_q * nb
                per = -(-U // sms)
                P = -(-U // per)
                assert P <= min(sms, U)
                sizes = [_bal_begin(p + 1, U, P) - _bal_begin(p, U, P) for p in range(P)]
                assert max(sizes) == per and max(sizes) - min(sizes) <= 1
                seen = {}
                for p in range(P):
                    u0, u1 = _bal_begin(p, U, P), _bal_begin(p + 1, U, P)
                    jobs = list(range(u0 // nb, (u1 - 1) // nb + 1))
                    for j, t in enumerate(jobs):
                        b0, b1 = max(u0, t * nb) - t * nb, min(u1, (t + 1) * nb) - t * nb
                        assert 0 <= b0 < b1 <= nb
                        if not (b0 == 0 and b1 == nb):
                            assert j in (0, len(jobs) - 1)
                        for blk in range(b0, b1):
                            assert (t, blk) not in seen
                            seen[(t, blk)] = p
                assert len(seen) == U


def test_balanced_schedule_choice_examples():
    # the balanced schedule only on request (measured slower than the uniform grid
    # at every s_q from 96 to 384 on 152 SMs)
    for s_q in (96, 160, 200, 250, 300, 384):
        assert b.mla_decode_plan(s_q, 640, num_sms=152).balanced_ctas == 0
    assert b.mla_decode_plan(96, 640, num_sms=152, force_splits=-1).balanced_ctas == 152
    assert b.mla_decode_plan(384, 640, num_sms=152, force_splits=-1).balanced_ctas == 152
    # s_q = 1, 16: the grid already spreads as evenly (10 x 1 block, 80 x 2 blocks)
    assert b.mla_decode_plan(1, 640, num_sms=152).balanced_ctas == 0
    assert b.mla_decode_plan(16, 640, num_sms=152).balanced_ctas == 0
    assert b.mla_decode_plan(96, 640, num_sms=152, force_splits=1).balanced_ctas == 0


def test_bf16_partials_setter_recomputes_the_workspace():
    ru = lambda x: -(-x // 256) * 256
    p = b.mla_decode_plan(16, 640, num_sms=152, force_splits=8)
    assert p.partial_bf16 == 0
    assert p.o_acc_bytes == 8 * 16 * 64 * 512 * 4
    b.mla_plan_set_partials_bf16(p)
    assert p.partial_bf16 == 1
    assert p.o_acc_bytes == 8 * 16 * 64 * 512 * 2
    assert p.lse_acc_offset == ru(p.o_acc_bytes)
    assert p.lse_acc_bytes == 8 * 16 * 64 * 4
    assert p.workspace_bytes == ru(p.lse_acc_offset + p.lse_acc_bytes)
    b.mla_plan_set_partials_bf16(p, False)
    assert bytes(p) == bytes(b.mla_decode_plan(16, 640, num_sms=152, force_splits=8))
    # one split: still no workspace; balanced: the slots' area in bf16
    p1 = b.mla_plan_set_partials_bf16(b.mla_decode_plan(96, 640, num_sms=152))
    assert p1.num_splits == 1 and p1.workspace_bytes == 0
    pb = b.mla_decode_plan(96, 640, num_sms=152, force_splits=-1)
    slots = balanced_slots(96, 10, 152)
    b.mla_plan_set_partials_bf16(pb)
    assert pb.workspace_bytes == ru(ru(slots * 96 * 64 * 512 * 2) + slots * 96 * 64 * 4)


def test_bf16_partials_setter_errors():
    invalid_arg = 1
    p = b.mla_decode_plan(16, 640, num_sms=152)
    before = bytes(p)
    with pytest.raises(b.SplitKVError) as e:
        b.mla_plan_set_partials_bf16(p, 2)
    assert e.value.status == invalid_arg
    assert bytes(p) == before                      # refused: the plan is left as it was
    assert b.lib().mla_plan_set_partials_bf16(None, 1) == invalid_arg
    q = b.MlaPlan()   # not made by mla_decode_plan
    assert b.lib().mla_plan_set_partials_bf16(ctypes.byref(q), 1) == invalid_arg


def test_package_reexports_every_entry_point():
    import split_kv_sparse_gb300 as pkg
    for name in b.EXPORTS:
        if name == "mla_status_string":
            continue      # wrapped as status_string
        assert hasattr(pkg, name), name


def test_index_check_switch_arguments():
    """mla_set_index_checks takes 0 or 1 only (no GPU needed: it sets a process-wide flag)."""
    for bad in (2, -1):
        with pytest.raises(b.SplitKVError) as e:
            b.mla_set_index_checks(bad)
        assert e.value.status == 1          # MLA_ERR_INVALID_ARG
    b.mla_set_index_checks(False)

"""Pins for the sparse-MLA oracle, each against something other than the oracle itself.

* torch's fp64 scaled_dot_product_attention (a library routine): with the
  gathered rows as keys, sparse MLA is multi-query attention with one KV head
  (K = rows, V = their first 512 dims). The sink is an extra key of score
  sink_h and V = 0, given to SDPA through an additive mask.
* torch.logsumexp for the log2-space LSE.
* closed forms: one index returns its V row; Q = 0 returns the mean of the
  gathered V rows with LSE2 = log2 |J|; a duplicated index counts twice; a
  -inf sink changes nothing; one index with a sink is scaled by 1/(1 + e^(sink - s)).
* split invariance: the combine of any split count equals the unsplit result.
* the workspace sizes printed in FlashMLA PR #25, "Measured" (tests/golden).
* planted mistakes in the oracle fail at least one of these pins.
"""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle.mla as om
from split_kv_sparse_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _small(seed=0, s_q=3, n_kv=300, topk=200, h=8, d_qk=40, d_v=32, pad=False):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((s_q, h, d_qk))
    kv = rng.standard_normal((n_kv, d_qk))
    idx = np.stack([rng.choice(n_kv, topk, replace=False) for _ in range(s_q)])
    if pad:
        for t in range(s_q):
            n = rng.integers(1, topk + 1)
            idx[t, n:] = -1
    return q, kv, idx.astype(np.int64), d_v


def _sdpa_ref(q, kv, idx, scale, d_v, sink=None):
    """torch fp64 SDPA per token over the valid gathered rows (+ an optional sink key)."""
    qt = torch.from_numpy(q)
    kvt = torch.from_numpy(kv)
    outs, lses = [], []
    for t in range(q.shape[0]):
        sel = idx[t][(idx[t] >= 0) & (idx[t] < kv.shape[0])]
        K = kvt[sel]
        V = kvt[sel, :d_v]
        h = q.shape[1]
        mask = None
        if sink is not None:
            K = torch.cat([K, torch.zeros(1, K.shape[1], dtype=K.dtype)])
            V = torch.cat([V, torch.zeros(1, V.shape[1], dtype=V.dtype)])
            mask = torch.zeros(1, h, 1, K.shape[0], dtype=torch.float64)
            mask[0, :, 0, -1] = torch.from_numpy(np.asarray(sink, dtype=np.float64))
        o = F.scaled_dot_product_attention(
            qt[t][None, :, None, :], K[None, None].expand(1, h, -1, -1),
            V[None, None].expand(1, h, -1, -1), attn_mask=mask, scale=scale)
        outs.append(o[0, :, 0].numpy())
        scores = scale * (qt[t] @ kvt[sel].T)
        lses.append((torch.logsumexp(scores, dim=-1) / math.log(2)).numpy())
    return np.stack(outs), np.stack(lses)


@pytest.mark.parametrize("seed,pad", [(0, False), (1, True), (2, False)])
def test_attention_matches_torch_sdpa(seed, pad):
    q, kv, idx, d_v = _small(seed, pad=pad)
    scale = 1.0 / math.sqrt(q.shape[-1])
    O, L = om.attention(q, kv, idx, scale, d_v)
    Or, Lr = _sdpa_ref(q, kv, idx, scale, d_v)
    np.testing.assert_allclose(O, Or, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(L, Lr, rtol=0, atol=1e-12)


def test_sink_matches_torch_sdpa_extra_key():
    q, kv, idx, d_v = _small(3)
    scale = 0.2
    sink = np.random.default_rng(9).standard_normal(q.shape[1]) * 2
    O, L = om.attention(q, kv, idx, scale, d_v, sink=sink)
    Or, Lr = _sdpa_ref(q, kv, idx, scale, d_v, sink=sink)
    np.testing.assert_allclose(O, Or, rtol=1e-12, atol=1e-13)
    # the returned LSE excludes the sink
    np.testing.assert_allclose(L, Lr, atol=1e-12)


def test_full_index_list_is_mqa_at_production_shape():
    """T = every row in order: sparse MLA == MQA over the whole cache (h=64, d_qk=576, d_v=512)."""
    inp = wl.mla_inputs(2, 700, 640, seed=5, index_mode="uniform")
    q = inp.q.double().numpy()
    kv = inp.kv.double().numpy()
    idx = np.tile(np.arange(700), (2, 1))
    O, L = om.attention(q, kv, idx, inp.sm_scale, 512)
    Or, Lr = _sdpa_ref(q, kv, idx, inp.sm_scale, 512)
    np.testing.assert_allclose(O, Or, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(L, Lr, atol=1e-11)


def test_single_index_returns_its_row():
    q, kv, _, d_v = _small(4)
    j = 17
    idx = np.full((q.shape[0], 5), -1)
    idx[:, 2] = j
    scale = 0.3
    O, L = om.attention(q, kv, idx, scale, d_v)
    for t in range(q.shape[0]):
        np.testing.assert_array_equal(O[t], np.broadcast_to(kv[j, :d_v], O[t].shape))
        s = scale * q[t] @ kv[j]
        np.testing.assert_allclose(L[t], s / math.log(2), atol=1e-13)


def test_single_index_with_sink_closed_form():
    q, kv, _, d_v = _small(5)
    idx = np.array([[42]] * q.shape[0])
    sink = np.linspace(-3, 3, q.shape[1])
    scale = 0.25
    O, _ = om.attention(q, kv, idx, scale, d_v, sink=sink)
    for t in range(q.shape[0]):
        s = scale * q[t] @ kv[42]
        w = 1.0 / (1.0 + np.exp(sink - s))
        np.testing.assert_allclose(O[t], w[:, None] * kv[42, :d_v][None], rtol=1e-13)


def test_zero_query_gives_mean_and_log2_count():
    _, kv, idx, d_v = _small(6, pad=True)
    q = np.zeros((idx.shape[0], 4, kv.shape[1]))
    O, L = om.attention(q, kv, idx, 0.1, d_v)
    for t in range(idx.shape[0]):
        sel = idx[t][idx[t] >= 0]
        np.testing.assert_allclose(O[t], np.broadcast_to(kv[sel, :d_v].mean(0), O[t].shape), rtol=1e-12)
        np.testing.assert_allclose(L[t], math.log2(len(sel)), atol=1e-13)


def test_duplicate_index_counts_twice():
    q, kv, _, d_v = _small(7)
    idx = np.array([[3, 3]] * q.shape[0])
    O, L = om.attention(q, kv, idx, 0.5, d_v)
    for t in range(q.shape[0]):
        s = 0.5 * q[t] @ kv[3]
        np.testing.assert_allclose(L[t], s / math.log(2) + 1.0, atol=1e-13)
        np.testing.assert_allclose(O[t], np.broadcast_to(kv[3, :d_v], O[t].shape), rtol=1e-14)


def test_minus_inf_sink_is_a_no_op():
    q, kv, idx, d_v = _small(8)
    sink = np.full(q.shape[1], -np.inf)
    O1, L1 = om.attention(q, kv, idx, 0.2, d_v)
    O2, L2 = om.attention(q, kv, idx, 0.2, d_v, sink=sink)
    np.testing.assert_array_equal(O1, O2)
    np.testing.assert_array_equal(L1, L2)


def test_padding_is_the_same_as_removal_and_empty_is_zero():
    q, kv, idx, d_v = _small(9, pad=True)
    idx[0, :] = -1                      # token 0 has nothing to attend
    idx[1, 5] = kv.shape[0] + 7         # out-of-range index is masked too
    O, L = om.attention(q, kv, idx, 0.2, d_v, sink=np.ones(q.shape[1]))
    assert np.all(O[0] == 0) and np.all(np.isneginf(L[0]))
    for t in range(1, q.shape[0]):
        sel = idx[t][(idx[t] >= 0) & (idx[t] < kv.shape[0])]
        Ot, Lt = om.attention(q[t:t + 1], kv, sel[None], 0.2, d_v, sink=np.ones(q.shape[1]))
        np.testing.assert_allclose(O[t], Ot[0], rtol=1e-14)
        np.testing.assert_allclose(L[t], Lt[0], rtol=1e-14)


def test_index_order_does_not_matter():
    q, kv, idx, d_v = _small(10)
    perm = np.random.default_rng(0).permutation(idx.shape[1])
    O1, L1 = om.attention(q, kv, idx, 0.2, d_v)
    O2, L2 = om.attention(q, kv, idx[:, perm], 0.2, d_v)
    np.testing.assert_allclose(O1, O2, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(L1, L2, atol=1e-12)


def test_split_ranges_rule():
    for topk in [1, 63, 64, 65, 640, 1000, 2048]:
        n_blk = -(-topk // 64)
        for S in range(1, 20):
            r = om.split_row_ranges(topk, S)
            assert len(r) == S
            assert r[0][0] == 0 and r[-1][1] == topk
            for a, b in zip(r, r[1:]):
                assert a[1] == b[0]
            blocks = [-(-(b - a) // 64) for a, b in r]
            # near-equal, the remainder on the leading splits
            assert blocks == [n_blk // S + (1 if s < n_blk % S else 0) for s in range(S)]
    # the degenerate layout of 64 entries over 16 splits: one full split, fifteen empty
    r = om.split_row_ranges(64, 16)
    assert r[0] == (0, 64) and all(a == b for a, b in r[1:])


@pytest.mark.parametrize("pad", [False, True])
def test_split_invariance_every_split_count(pad):
    q, kv, idx, d_v = _small(11, topk=300, pad=pad)
    sink = np.random.default_rng(3).standard_normal(q.shape[1])
    O1, L1 = om.attention(q, kv, idx, 0.2, d_v, sink=sink)
    for S in range(1, 17):                               # includes S > n_blk (= 5)
        O, L = om.decode(q, kv, idx, 0.2, S, sink=sink, d_v=d_v)
        np.testing.assert_allclose(O, O1, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(L, L1, atol=1e-12)


def test_empty_splits_are_zero_and_minus_inf_and_drop_out():
    q, kv, idx, d_v = _small(12, topk=64)
    O_s, L_s = om.split_partials(q, kv, idx, 0.2, 16, d_v)
    assert np.all(O_s[1:] == 0) and np.all(np.isneginf(L_s[1:]))
    O1, L1 = om.combine(O_s[:1], L_s[:1])
    O16, L16 = om.combine(O_s, L_s)
    np.testing.assert_array_equal(O1, O16)
    np.testing.assert_array_equal(L1, L16)


def test_combine_all_empty():
    O, L = om.combine(np.zeros((4, 2, 3, 5)), np.full((4, 2, 3), -np.inf), sink=np.zeros(3))
    assert np.all(O == 0) and np.all(np.isneginf(L))


def test_partials_are_normalised_per_split():
    """Each partial is a convex combination of its own V rows (weights sum to 1)."""
    q, kv, idx, d_v = _small(13, topk=256)
    kv = kv.copy()
    kv[:, :d_v] = 1.0                                    # every V row is all ones
    O_s, L_s = om.split_partials(q, kv, idx, 0.3, 4, d_v)
    np.testing.assert_allclose(O_s, 1.0, rtol=1e-13)


def test_workspace_bytes_match_page():
    with open(os.path.join(GOLDEN, "workspace_bytes.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    assert len(rows) == 2
    for S, s_q, h, d_v, mb in rows:
        b = om.workspace_bytes(int(S), int(s_q), int(h), int(d_v))
        assert round(b / 1e6, 2 if float(mb) < 10 else 1) == float(mb)
    assert om.workspace_bytes(8, 1) == 1048576
    assert om.workspace_bytes(8, 16) == 16777216


# ---- planted mistakes: each must fail at least one pin above -------------------------

def _pins_pass():
    try:
        test_attention_matches_torch_sdpa(0, False)
        test_sink_matches_torch_sdpa_extra_key()
        test_single_index_with_sink_closed_form()
        test_split_invariance_every_split_count(True)
        test_empty_splits_are_zero_and_minus_inf_and_drop_out()
        test_partials_are_normalised_per_split()
    except AssertionError:
        return False
    return True


def test_pins_pass_on_unmodified_oracle():
    assert _pins_pass()


@pytest.mark.parametrize("planted", ["log_base", "remainder_last", "combine_exp_base",
                                     "sink_in_partials", "drop_sink"])
def test_planted_oracle_mistakes_are_caught(monkeypatch, planted):
    if planted == "log_base":
        monkeypatch.setattr(om, "LN2", math.log(10.0))
    elif planted == "remainder_last":
        orig = om.split_row_ranges
        monkeypatch.setattr(om, "split_row_ranges",
                            lambda topk, S, unit=64: [(a + 1 if a else a, b) for a, b in orig(topk, S, unit)])
    elif planted == "combine_exp_base":
        monkeypatch.setattr(om.np, "exp2", np.exp)
    elif planted == "sink_in_partials":
        orig_att = om.attention
        monkeypatch.setattr(om, "attention", lambda q, kv, idx, sc, d_v=512, sink=None, cols=None:
                            orig_att(q, kv, idx, sc, d_v, sink=np.zeros(np.shape(q)[1]), cols=cols)
                            if cols is not None else orig_att(q, kv, idx, sc, d_v, sink, cols))
    elif planted == "drop_sink":
        orig_att = om.attention
        monkeypatch.setattr(om, "attention", lambda q, kv, idx, sc, d_v=512, sink=None, cols=None:
                            orig_att(q, kv, idx, sc, d_v, None, cols))
    assert not _pins_pass()

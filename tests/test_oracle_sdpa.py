"""Pins for the dense FP8 split-KV SDPA oracle.

* torch's fp64 scaled_dot_product_attention with an explicit bottom-right
  causal mask and repeat_interleave of the KV heads (GQA), on the dequantised
  codes (a library routine independent of the oracle);
* the chunk rule (near-equal tiles, remainder to the leading splits; a chunk
  past the end is empty and gives O = 0 / LSE = -inf);
* split invariance for every split count;
* closed forms: a sequence with one key returns that key's V row; amax is
  the largest |O|.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle.sdpa as osd
from oracle import codecs
from split_kv_sparse_gb300 import workloads as wl


def _small(seed=0, batch=3, h_q=8, h_kv=2, d=32, q_per_seq=(1, 5), kv_len=(40, 300)):
    return wl.sdpa_inputs(batch, h_q, h_kv, d, q_per_seq=q_per_seq, kv_len=kv_len, seed=seed)


def _torch_ref(inp):
    q = torch.from_numpy(codecs.e4m3_decode(inp.q.numpy()) * inp.descale_q)
    k = torch.from_numpy(codecs.e4m3_decode(inp.k.numpy()) * inp.descale_k)
    v = torch.from_numpy(codecs.e4m3_decode(inp.v.numpy()) * inp.descale_v)
    cq, ck = inp.cu_seqlens_q.tolist(), inp.cu_seqlens_kv.tolist()
    outs, lses = [], []
    g = inp.h_q // inp.h_kv
    for b in range(inp.batch):
        qs = q[cq[b]:cq[b + 1]].transpose(0, 1)                      # [h_q, sq, d]
        ks = k[ck[b]:ck[b + 1]].transpose(0, 1).repeat_interleave(g, 0)
        vs = v[ck[b]:ck[b + 1]].transpose(0, 1).repeat_interleave(g, 0)
        sq, skv = qs.shape[1], ks.shape[1]
        allowed = torch.arange(skv)[None, :] <= (skv - sq + torch.arange(sq))[:, None]
        o = F.scaled_dot_product_attention(qs[None], ks[None], vs[None], attn_mask=allowed[None, None],
                                           scale=inp.sm_scale)
        outs.append(o[0].transpose(0, 1))
        s = inp.sm_scale * qs @ ks.transpose(1, 2)
        s = s.masked_fill(~allowed[None], -math.inf)
        lses.append((torch.logsumexp(s, -1) / math.log(2)).transpose(0, 1))
    return torch.cat(outs).numpy(), torch.cat(lses).numpy()


@pytest.mark.parametrize("seed", [0, 1])
def test_matches_torch_sdpa_causal_gqa(seed):
    inp = _small(seed)
    O, L = osd.attention(inp)
    Or, Lr = _torch_ref(inp)
    np.testing.assert_allclose(O, Or, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(L, Lr, atol=1e-11)


def test_chunk_rule():
    for kv_len in [1, 127, 128, 129, 1024, 16384, 5000]:
        n = -(-kv_len // 128)
        for S in range(1, 18):
            r = osd.chunk_ranges(kv_len, S)
            assert r[0][0] == 0 and r[-1][1] == kv_len
            assert all(a[1] == b[0] for a, b in zip(r, r[1:]))
            tiles = [-(-(b - a) // 128) for a, b in r]
            assert tiles == [n // S + (1 if s < n % S else 0) for s in range(S)]


@pytest.mark.parametrize("S", [1, 2, 3, 5, 8, 16])
def test_split_invariance(S):
    inp = _small(2, kv_len=(100, 700))
    O1, L1 = osd.attention(inp)
    O, L, amax = osd.decode(inp, S)
    np.testing.assert_allclose(O, O1, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(L, L1, atol=1e-12)
    assert amax == np.max(np.abs(O1)) or math.isclose(amax, np.max(np.abs(O1)), rel_tol=1e-12)


def test_empty_chunks_past_the_end():
    inp = _small(3, kv_len=(50, 120))           # every sequence fits in one 128-key tile
    O_s, L_s = osd.split_partials(inp, 4)
    assert np.all(O_s[1:] == 0) and np.all(np.isneginf(L_s[1:]))


def test_single_key_returns_its_value_row():
    inp = _small(4, q_per_seq=(1, 1), kv_len=(1, 1))
    O, L = osd.attention(inp)
    v = codecs.e4m3_decode(inp.v.numpy()) * inp.descale_v
    g = inp.h_q // inp.h_kv
    for b in range(inp.batch):
        for j in range(inp.h_q):
            np.testing.assert_array_equal(O[b, j], v[b, j // g])


def test_planted_causal_offset_is_caught(monkeypatch):
    """Top-left (instead of bottom-right) causal alignment fails the library pin."""
    orig = osd._attend_rows
    monkeypatch.setattr(osd, "_attend_rows",
                        lambda q, K, V, sc, lo, hi, pos: orig(q, K, V, sc, lo, hi, pos - pos[0]))
    inp = _small(5)
    O, _ = osd.attention(inp)
    Or, _ = _torch_ref(inp)
    assert not np.allclose(O, Or, rtol=1e-6)


def test_planted_gqa_mapping_is_caught(monkeypatch):
    inp = _small(6)
    Or, _ = _torch_ref(inp)
    inp.h_kv = inp.h_q // 2 if inp.h_q // 2 != inp.h_kv else inp.h_kv // 2  # wrong group size
    try:
        O, _ = osd.attention(inp)
    except IndexError:
        return
    assert not np.allclose(O, Or, rtol=1e-6)

"""fp64 oracle for dense split-KV FP8 SDPA decode (test infrastructure only).

The form is the one cuDNN-frontend PR #768 describes for its SM107/SM120 FP8
forward kernels ("Conversation", both commit messages):
  * per-tensor scaled FP8 e4m3 Q/K/V; a bf16 O;
  * each Q tile's (already masked) KV range is cut into SPLIT_KV near-equal
    chunks with the remainder going to the leading splits; a chunk past the
    end is empty and enters the combine as O := 0 / LSE := -inf;
  * partial O and per-split LSE are written into split-major slots and a
    combine folds them; the combine owns the amax of the recombined O,
    because a max over partials over-reports it.

Readings where the page is silent (each listed in the design notes):
  - values are code * descale per tensor; scores s = sm_scale * q . k in
    natural-log units, sm_scale = 1/sqrt(d);
  - GQA: query head j reads KV head j // (h_q / h_kv);
  - causal alignment is bottom-right: query i of a sequence with s_q new
    tokens and kv_len keys sits at position kv_len - s_q + i and sees keys
    0..that position;
  - the chunk unit is a tile of 128 keys over [0, kv_len).
"""
from __future__ import annotations

from typing import List, Tuple

import numpy as np

from . import codecs
from .mla import LN2, _i64, combine

KEY_TILE = 128


def _dequant(codes, descale: float) -> np.ndarray:
    try:
        import torch
        if isinstance(codes, torch.Tensor):
            codes = codes.detach().cpu().view(torch.uint8).numpy()
    except ImportError:  # pragma: no cover
        pass
    return codecs.e4m3_decode(np.asarray(codes, dtype=np.uint8)) * descale


def chunk_ranges(kv_len: int, num_splits: int, unit: int = KEY_TILE) -> List[Tuple[int, int]]:
    """Key range [k0, k1) of each split: near-equal tile counts, remainder to the leading splits."""
    n_tiles = -(-kv_len // unit)
    base, rem = divmod(n_tiles, num_splits)
    out, b = [], 0
    for s in range(num_splits):
        cnt = base + (1 if s < rem else 0)
        out.append((min(b * unit, kv_len), min((b + cnt) * unit, kv_len)))
        b += cnt
    return out


def _attend_rows(q, K, V, sm_scale, key_lo, key_hi, pos):
    """Queries q [n, d] at positions pos [n] over keys [key_lo, key_hi) of K/V,
    each query limited to keys <= its position. Returns (O [n, d], LSE2 [n]);
    a query with no key gives (0, -inf)."""
    n = q.shape[0]
    O = np.zeros((n, V.shape[1]))
    L = np.full(n, -np.inf)
    if key_hi <= key_lo:
        return O, L
    keys = np.arange(key_lo, key_hi)
    has = key_lo <= pos
    if not has.any():
        return O, L
    s = sm_scale * (q @ K[key_lo:key_hi].T)                  # [n, keys]
    s = np.where(keys[None, :] <= pos[:, None], s, -np.inf)
    m = np.where(has, s.max(axis=1), 0.0)
    e = np.exp(s - m[:, None])
    z = e.sum(axis=1)
    with np.errstate(invalid="ignore", divide="ignore"):
        O = np.where(has[:, None], (e @ V[key_lo:key_hi]) / z[:, None], 0.0)
        L = np.where(has, (m + np.log(z)) / LN2, -np.inf)
    return O, L


def _run(inp, num_splits: int):
    qv = _dequant(inp.q, inp.descale_q)
    kv_ = _dequant(inp.k, inp.descale_k)
    vv = _dequant(inp.v, inp.descale_v)
    cu_q = _i64(inp.cu_seqlens_q)
    cu_k = _i64(inp.cu_seqlens_kv)
    total_q, h_q, d = qv.shape
    group = h_q // inp.h_kv
    O_s = np.zeros((num_splits, total_q, h_q, d))
    L_s = np.full((num_splits, total_q, h_q), -np.inf)
    for b in range(len(cu_q) - 1):
        q0, q1 = int(cu_q[b]), int(cu_q[b + 1])
        k0, k1 = int(cu_k[b]), int(cu_k[b + 1])
        sq, skv = q1 - q0, k1 - k0
        pos = skv - sq + np.arange(sq)
        ranges = chunk_ranges(skv, num_splits)
        for j in range(h_q):
            g = j // group
            K = kv_[k0:k1, g]
            V = vv[k0:k1, g]
            for s, (lo, hi) in enumerate(ranges):
                O_s[s, q0:q1, j], L_s[s, q0:q1, j] = _attend_rows(qv[q0:q1, j], K, V,
                                                                  inp.sm_scale, lo, hi, pos)
    return O_s, L_s


def split_partials(inp, num_splits: int):
    """Per-split partial O [S, total_q, h_q, d] (normalised per split) and LSE2 [S, total_q, h_q]."""
    return _run(inp, num_splits)


def attention(inp):
    """Unsplit result (O [total_q, h_q, d], LSE2 [total_q, h_q]) by the definition."""
    O_s, L_s = _run(inp, 1)
    return O_s[0], L_s[0]


def decode(inp, num_splits: int = 1):
    """Split partials folded by the log-sum-exp combine; returns (O, LSE2, amax of O)."""
    O_s, L_s = _run(inp, num_splits)
    O, L = combine(O_s, L_s, None)
    return O, L, float(np.max(np.abs(O))) if O.size else 0.0

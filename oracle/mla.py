"""fp64 oracle for split-KV sparse-MLA decode (test infrastructure only).

What the path computes, as read from the pages:

* FlashMLA PR #25, "Purpose": each decode (query) token has h_q = 64 heads
  that attend over a top-k set of rows of one shared latent KV cache
  ("topk 128+512"). A row has d_qk = 576 dims (512 latent + 64 RoPE); V is the
  first 512 dims of the same row.
* FlashMLA PR #25, "What changes": the work is cut into (query token, KV
  split) jobs; each job walks only its own KV block range and stores an fp32
  partial O normalised by that split's l_i plus a log2-space LSE; the
  attention sink is left to the combine.
* "The Split-K Dispatch", "The LSE Combine Strategy": the combine takes the
  global max of the per-split maxima and weights every split by
  exp2(local - global) before dividing by the corrected denominator.
* cuDNN-frontend PR #768, SM120 FP8 commit: chunks are near-equal with the
  remainder going to the leading splits; a chunk past the end is empty and
  enters the combine as O := 0 / LSE := -inf.

Readings where the pages are silent (each listed in the design notes):
  - scores s_j = sm_scale * <q_h, kv_j> in natural-log units; "log2-space LSE"
    is log2(sum_j exp(s_j)); both the partial and the final LSE are log2.
  - the sink is a per-head logit in the same natural-log units; it adds
    exp(sink_h) to the softmax denominator, carries no V, and the returned LSE
    excludes it. An empty row set gives O = 0 and LSE = -inf with or without a sink.
  - an index outside [0, n_kv) (e.g. the -1 padding) is masked; valid indices
    count with multiplicity.
  - the split unit is a block of 64 top-k entries: n_blk = ceil(topk / 64);
    split s owns floor(n_blk / S) + (s < n_blk mod S) consecutive blocks.

Everything is computed in float64 from the exact bf16 input values; matmuls
and sums use numpy as library steps, with no blocking or reordering beyond the
definitions above.
"""
from __future__ import annotations

import math
from typing import List, Optional, Tuple

import numpy as np

from . import codecs

LN2 = math.log(2.0)
SPLIT_UNIT = 64  # top-k entries per KV block (the split granularity)


def _f64(x) -> np.ndarray:
    """torch tensor / array -> float64 numpy array (bf16 -> fp64 is exact)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


def _i64(x) -> np.ndarray:
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu", torch.int64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.int64)


def attention(q, kv, idx, sm_scale: float, d_v: int = 512, sink=None,
              cols: Optional[Tuple[int, int]] = None):
    """Sparse-MLA decode attention by its definition.

    q: [s_q, h, d_qk]; kv: [n_kv, d_qk]; idx: [s_q, topk] integer rows.
    cols: optional (c0, c1) restricting each token to top-k entries c0..c1-1
    (used for one split's range). sink: optional [h] logits.

    Returns (O [s_q, h, d_v] float64, LSE2 [s_q, h] float64) with
      J    = valid entries of idx[t, c0:c1] (0 <= idx < n_kv), with multiplicity
      s_j  = sm_scale * q[t, h] . kv[idx_j]
      LSE2 = log2(sum_j exp(s_j))                          (-inf if J is empty)
      O    = sum_j exp(s_j) kv[idx_j, :d_v] / (sum_j exp(s_j) + exp(sink_h))
    """
    q = _f64(q)
    kv = _f64(kv)
    idx = _i64(idx)
    s_q, h, _ = q.shape
    n_kv = kv.shape[0]
    c0, c1 = cols if cols is not None else (0, idx.shape[1])
    sink = None if sink is None else _f64(sink)
    O = np.zeros((s_q, h, d_v))
    LSE = np.full((s_q, h), -np.inf)
    for t in range(s_q):
        row = idx[t, c0:c1]
        sel = row[(row >= 0) & (row < n_kv)]
        if sel.size == 0:
            continue
        K = kv[sel]                            # [J, d_qk]
        V = kv[sel, :d_v]                      # [J, d_v]
        s = sm_scale * (q[t] @ K.T)            # [h, J], natural-log units
        m = s.max(axis=1)                      # shift for a stable exp
        e = np.exp(s - m[:, None])
        z = e.sum(axis=1)                      # sum_j exp(s_j - m)
        LSE[t] = (m + np.log(z)) / LN2
        denom = z.copy()
        if sink is not None:
            denom = denom + np.exp(sink - m)
        O[t] = (e @ V) / denom[:, None]
    return O, LSE


def split_row_ranges(topk: int, num_splits: int, unit: int = SPLIT_UNIT) -> List[Tuple[int, int]]:
    """Top-k entry range [r0, r1) of every split.

    n_blk = ceil(topk / unit) blocks; split s gets floor(n_blk / S) blocks plus
    one more if s < n_blk mod S, consecutively from the start; a split with no
    block gets an empty range (cuDNN-frontend PR #768, SM120 FP8 commit).
    """
    if num_splits < 1:
        raise ValueError("num_splits must be >= 1")
    n_blk = -(-topk // unit)
    base, rem = divmod(n_blk, num_splits)
    out = []
    b = 0
    for s in range(num_splits):
        cnt = base + (1 if s < rem else 0)
        out.append((min(b * unit, topk), min((b + cnt) * unit, topk)))
        b += cnt
    return out


def split_partials(q, kv, idx, sm_scale: float, num_splits: int, d_v: int = 512):
    """Per-split fp32-protocol partials, computed in fp64.

    Returns (O_s [S, s_q, h, d_v], LSE_s [S, s_q, h]): O_s is the split's output
    normalised by its own sum (no sink), LSE_s its log2-space LSE; an empty
    split gives (0, -inf) (FlashMLA PR #25, "What changes").
    """
    idx = _i64(idx)
    s_q, h = _f64(q).shape[:2]
    ranges = split_row_ranges(idx.shape[1], num_splits)
    O_s = np.zeros((num_splits, s_q, h, d_v))
    L_s = np.full((num_splits, s_q, h), -np.inf)
    for s, (r0, r1) in enumerate(ranges):
        if r1 > r0:
            O_s[s], L_s[s] = attention(q, kv, idx, sm_scale, d_v, sink=None, cols=(r0, r1))
    return O_s, L_s


def combine(O_s, LSE_s, sink=None):
    """Log-sum-exp fold of split partials ("The Split-K Dispatch", "The LSE Combine Strategy").

      M   = max_s LSE_s
      w_s = 2**(LSE_s - M)                       (0 for an empty split)
      O   = sum_s w_s O_s / (sum_s w_s + exp(sink_h) / 2**M)
      LSE = M + log2(sum_s w_s)
    A (token, head) with every split empty gives O = 0, LSE = -inf.
    The sink enters here and only here (FlashMLA PR #25, "What changes").
    """
    O_s = np.asarray(O_s, dtype=np.float64)
    L = np.asarray(LSE_s, dtype=np.float64)
    M = L.max(axis=0)
    empty = np.isneginf(M)
    Msafe = np.where(empty, 0.0, M)
    w = np.where(np.isneginf(L), 0.0, np.exp2(L - Msafe[None]))
    wsum = w.sum(axis=0)
    num = (w[..., None] * O_s).sum(axis=0)
    denom = wsum.copy()
    if sink is not None:
        sink = _f64(sink)
        denom = denom + np.exp(sink[None, :] - Msafe * LN2)
    with np.errstate(invalid="ignore", divide="ignore"):
        O = np.where(empty[..., None], 0.0, num / denom[..., None])
        LSE = np.where(empty, -np.inf, Msafe + np.log2(wsum))
    return O, LSE


def cast_output(O, out_dtype: str, inv_scale: float = 1.0):
    """Final output cast. Returns (values as float64, raw codes or None).

    "f32": round to float32 (the parity pass-through); "bf16": RNE to bf16;
    "e4m3": RNE + saturate of O * inv_scale to FP8 e4m3 (dequantised as code * scale).
    """
    O = np.asarray(O, dtype=np.float64)
    if out_dtype == "f32":
        v = O.astype(np.float32).astype(np.float64)
        return v, None
    if out_dtype == "bf16":
        return codecs.bf16_round(O), codecs.bf16_bits(O)
    if out_dtype == "e4m3":
        y = O * inv_scale
        return codecs.e4m3_round(y), codecs.e4m3_encode(y)
    raise ValueError(out_dtype)


def amax(O) -> float:
    """Largest |O| of the recombined, pre-cast output (cuDNN-frontend PR #768:
    the combine owns the amax of the recombined O)."""
    O = np.asarray(O, dtype=np.float64)
    return float(np.max(np.abs(O))) if O.size else 0.0


def workspace_bytes(num_splits: int, s_q: int, h_q: int = 64, d_v: int = 512) -> int:
    """Partial-O bytes per layer per step: num_splits * s_q * h_q * d_v * 4
    (FlashMLA PR #25, "Measured": 1.05 MB at one token / 8 splits, 16.8 MB at 16 tokens)."""
    return num_splits * s_q * h_q * d_v * 4


def decode(q, kv, idx, sm_scale: float, num_splits: int = 1, sink=None, d_v: int = 512):
    """The whole path as the split method computes it: partials, then the combine."""
    O_s, L_s = split_partials(q, kv, idx, sm_scale, num_splits, d_v)
    return combine(O_s, L_s, sink)

"""Seeded synthetic workloads for split-KV sparse-MLA decode and dense FP8 SDPA decode.

This module only draws inputs. It holds none of the attention arithmetic, so
both the CUDA path and the fp64 oracle can consume the same tensors without
sharing any of the computation.

Shapes follow the pages' workloads:
  * FlashMLA PR #25, "Purpose" and "Measured": h_q = 64 query heads per
    decode token attending over top-k = 128 + 512 rows of one latent KV cache
    (d_qk = 576 = 512 latent + 64 RoPE dims; V = the first 512 dims).
  * cuDNN-frontend PR #768 (SM120 FP8 commit): dense FP8 SDPA, per-tensor
    scaled e4m3 Q/K/V, bf16 O, ragged batches.

All draws use numpy's PCG64 generator with an explicit seed; floating-point
values are drawn in float32 and rounded once to bf16 by torch (round to
nearest even), so the bf16 tensors are the exact inputs both sides see.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

H_Q = 64
D_QK = 576
D_V = 512
MLA_SM_SCALE = 1.0 / math.sqrt(D_QK)


@dataclass
class MlaInputs:
    q: torch.Tensor            # bf16 [s_q, 64, 576]
    kv: torch.Tensor           # bf16 [n_kv, 576]
    idx: torch.Tensor          # int32 [s_q, topk]; -1 = padding
    sink: Optional[torch.Tensor]  # fp32 [64] natural-log logits, or None
    sm_scale: float

    @property
    def s_q(self) -> int:
        return self.q.shape[0]

    @property
    def topk(self) -> int:
        return self.idx.shape[1]

    @property
    def n_kv(self) -> int:
        return self.kv.shape[0]


def _bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def window_plus_uniform_indices(rng: np.random.Generator, s_q: int, n_kv: int,
                                window: int = 128, n_uniform: int = 512) -> np.ndarray:
    """Top-k rows shaped like the pages' "topk 128+512".

    Token t sits at position p_t = n_kv - s_q + t. Its first `window` entries
    are the rows [p_t - window + 1, p_t] in ascending order; the remaining
    `n_uniform` entries are distinct rows drawn uniformly from [0, p_t - window + 1).
    """
    out = np.empty((s_q, window + n_uniform), dtype=np.int32)
    for t in range(s_q):
        p = n_kv - s_q + t
        lo = p - window + 1
        if lo < n_uniform:
            raise ValueError("n_kv too small for the window + uniform structure")
        out[t, :window] = np.arange(lo, p + 1, dtype=np.int32)
        out[t, window:] = rng.choice(lo, size=n_uniform, replace=False).astype(np.int32)
    return out


def uniform_distinct_indices(rng: np.random.Generator, s_q: int, n_kv: int, topk: int) -> np.ndarray:
    out = np.empty((s_q, topk), dtype=np.int32)
    for t in range(s_q):
        out[t] = rng.choice(n_kv, size=topk, replace=False).astype(np.int32)
    return out


def padded_indices(rng: np.random.Generator, s_q: int, n_kv: int, topk: int) -> np.ndarray:
    """Per token a valid count uniform in [1, topk]; valid rows distinct and uniform, rest -1."""
    out = np.full((s_q, topk), -1, dtype=np.int32)
    for t in range(s_q):
        n = int(rng.integers(1, topk + 1))
        out[t, :n] = rng.choice(n_kv, size=n, replace=False).astype(np.int32)
    return out


def mla_inputs(s_q: int, n_kv: int, topk: int = 640, *, seed: int = 0,
               index_mode: str = "window", v_mean: float = 0.0,
               with_sink: bool = False, h_q: int = H_Q) -> MlaInputs:
    """Sparse-MLA decode inputs.

    index_mode: "window" (128 most recent rows + uniform rest), "uniform"
    (distinct uniform rows) or "padded" (valid count uniform in [1, topk], rest -1).
    v_mean: mean of the V dims (0..511) of every KV row; 1.0 gives the
    non-cancelling variant. The RoPE dims stay N(0, 1).
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    kv = rng.standard_normal((n_kv, D_QK), dtype=np.float32)
    if v_mean != 0.0:
        kv[:, :D_V] += np.float32(v_mean)
    q = rng.standard_normal((s_q, h_q, D_QK), dtype=np.float32)
    if index_mode == "window":
        idx = window_plus_uniform_indices(rng, s_q, n_kv, 128, topk - 128)
    elif index_mode == "uniform":
        idx = uniform_distinct_indices(rng, s_q, n_kv, topk)
    elif index_mode == "padded":
        idx = padded_indices(rng, s_q, n_kv, topk)
    else:
        raise ValueError(index_mode)
    sink = torch.from_numpy(rng.standard_normal(h_q, dtype=np.float32)) if with_sink else None
    return MlaInputs(q=_bf16(q), kv=_bf16(kv), idx=torch.from_numpy(idx), sink=sink,
                     sm_scale=1.0 / math.sqrt(D_QK))


def mla_queries(s_q: int, n_kv: int, topk: int = 640, *, seed: int = 0, h_q: int = H_Q):
    """Queries and "128 + 512" indices of one decode step without a cache (for callers that
    bring their own cache, e.g. one per model layer): Q ~ N(0, 1) bf16 [s_q, h_q, 576] and
    int32 indices [s_q, topk] drawn as in mla_inputs's "window" mode."""
    rng = np.random.Generator(np.random.PCG64(seed))
    q = rng.standard_normal((s_q, h_q, D_QK), dtype=np.float32)
    idx = window_plus_uniform_indices(rng, s_q, n_kv, 128, topk - 128)
    return _bf16(q), torch.from_numpy(idx)


# --------------------------------------------------------------------------------------
# Dense FP8 GQA decode (cuDNN-frontend PR #768 form)
# --------------------------------------------------------------------------------------

@dataclass
class SdpaInputs:
    q: torch.Tensor        # uint8 e4m3 codes [total_q, h_q, d]
    k: torch.Tensor        # uint8 e4m3 codes [total_kv, h_kv, d]
    v: torch.Tensor        # uint8 e4m3 codes [total_kv, h_kv, d]
    descale_q: float
    descale_k: float
    descale_v: float
    cu_seqlens_q: torch.Tensor   # int32 [batch + 1]
    cu_seqlens_kv: torch.Tensor  # int32 [batch + 1]
    sm_scale: float
    h_q: int
    h_kv: int
    d: int

    @property
    def batch(self) -> int:
        return self.cu_seqlens_q.numel() - 1


def quantize_e4m3_per_tensor(x: np.ndarray):
    """Per-tensor scaled FP8 input prep: descale = amax / 448, code = e4m3(x / descale).

    Uses torch's float8_e4m3fn conversion (round to nearest even) on values
    already inside [-448, 448]; returns (uint8 codes, descale).
    """
    amax = float(np.max(np.abs(x)))
    descale = amax / 448.0 if amax > 0 else 1.0
    y = np.clip(x / np.float32(descale), -448.0, 448.0).astype(np.float32)
    codes = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, float(descale)


def sdpa_inputs(batch: int = 8, h_q: int = 32, h_kv: int = 8, d: int = 128, *,
                q_per_seq=(1, 16), kv_len=(1024, 16384), seed: int = 0) -> SdpaInputs:
    rng = np.random.Generator(np.random.PCG64(seed))
    sq = rng.integers(q_per_seq[0], q_per_seq[1] + 1, size=batch)
    skv = rng.integers(kv_len[0], kv_len[1] + 1, size=batch)
    skv = np.maximum(skv, sq)
    cu_q = np.concatenate([[0], np.cumsum(sq)]).astype(np.int32)
    cu_kv = np.concatenate([[0], np.cumsum(skv)]).astype(np.int32)
    q = rng.standard_normal((int(cu_q[-1]), h_q, d), dtype=np.float32)
    k = rng.standard_normal((int(cu_kv[-1]), h_kv, d), dtype=np.float32)
    v = rng.standard_normal((int(cu_kv[-1]), h_kv, d), dtype=np.float32)
    qc, dq = quantize_e4m3_per_tensor(q)
    kc, dk = quantize_e4m3_per_tensor(k)
    vc, dv = quantize_e4m3_per_tensor(v)
    return SdpaInputs(q=qc, k=kc, v=vc, descale_q=dq, descale_k=dk, descale_v=dv,
                      cu_seqlens_q=torch.from_numpy(cu_q), cu_seqlens_kv=torch.from_numpy(cu_kv),
                      sm_scale=1.0 / math.sqrt(d), h_q=h_q, h_kv=h_kv, d=d)

"""Why the path keeps P as bf16 hi + lo and the split partials in fp32.

Each cheaper choice is simulated on top of the oracle's fp64 arithmetic, with only
that one rounding added, and checked against the FP8-output rules the parity tests
apply (FlashMLA PR #25, "Test plan": FP8 codes compared after the same cast, every
code within one step of the oracle's, at least 99 % identical where V does not
cancel). The cheaper choice breaks a rule; the kept choice meets it. CPU only:
these tests use the oracle and the codecs, never the CUDA path.
"""
import numpy as np
import torch

from oracle import codecs
from oracle.mla import attention, combine, split_partials
from split_kv_sparse_gb300 import workloads as wl


def _code_order(codes: np.ndarray) -> np.ndarray:
    """Position of each e4m3 code on the number line (sign-magnitude -> integer)."""
    c = codes.astype(np.int64)
    mag = c & 0x7F
    return np.where((c >> 7) & 1, -mag, mag)


def _fp8_steps(O_test: np.ndarray, O_ref: np.ndarray, inv_scale: float = 64.0) -> np.ndarray:
    a = _code_order(codecs.e4m3_encode(O_test * inv_scale))
    b = _code_order(codecs.e4m3_encode(O_ref * inv_scale))
    return np.abs(a - b)


def _attention_with_rounded_p(inp, round_p):
    """The oracle's attention with the exponentials e_j = exp(s_j - max) passed through
    round_p before the P.V product; the denominator keeps the exact sum (as the kernel's
    fp32 row sums do)."""
    q = inp.q.double().numpy()
    kv = inp.kv.double().numpy()
    idx = inp.idx.numpy()
    sink = inp.sink.double().numpy() if inp.sink is not None else None
    O = np.zeros((q.shape[0], q.shape[1], 512))
    for t in range(q.shape[0]):
        sel = idx[t][(idx[t] >= 0) & (idx[t] < kv.shape[0])]
        K, V = kv[sel], kv[sel, :512]
        s = inp.sm_scale * (q[t] @ K.T)
        m = s.max(axis=1)
        e = np.exp(s - m[:, None])
        denom = e.sum(axis=1)
        if sink is not None:
            denom = denom + np.exp(sink - m)
        O[t] = (round_p(e) @ V) / denom[:, None]
    return O


def _single_bf16(e):
    return codecs.bf16_round(e.astype(np.float32).astype(np.float64))


def _hi_lo_bf16(e):
    f = e.astype(np.float32)
    hi = (f.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32)
    lo = codecs.bf16_round((f - hi).astype(np.float64))
    return hi.astype(np.float64) + lo


def test_single_bf16_p_breaks_the_one_step_fp8_rule():
    """Cancelling V (config 2, V ~ N(0,1)): a single bf16 P moves some FP8 codes by more than
    one step (near zero, where codes are dense); P_hi + P_lo keeps every code within one."""
    inp = wl.mla_inputs(6, 32768, 640, seed=31, v_mean=0.0, with_sink=True)
    O, _ = attention(inp.q, inp.kv, inp.idx, inp.sm_scale, sink=inp.sink)
    single = _attention_with_rounded_p(inp, _single_bf16)
    hilo = _attention_with_rounded_p(inp, _hi_lo_bf16)
    assert _fp8_steps(single, O).max() > 1
    assert _fp8_steps(hilo, O).max() <= 1
    rel = np.linalg.norm(hilo - O, axis=-1) / np.linalg.norm(O, axis=-1)
    assert rel.max() < 1e-5


def test_bf16_partials_break_the_identical_code_floor():
    """Non-cancelling V (V ~ N(1,1)), two splits: bf16 partials leave fewer than 99 % of the
    FP8 codes equal to the oracle's; fp32 partials (what the split pass stores) keep the floor."""
    inp = wl.mla_inputs(16, 32768, 640, seed=31, v_mean=1.0, with_sink=True)
    O, _ = attention(inp.q, inp.kv, inp.idx, inp.sm_scale, sink=inp.sink)
    O_s, L_s = split_partials(inp.q, inp.kv, inp.idx, inp.sm_scale, 2)
    as_bf16, _ = combine(codecs.bf16_round(O_s.astype(np.float32).astype(np.float64)), L_s, sink=inp.sink)
    as_fp32, _ = combine(O_s.astype(np.float32).astype(np.float64), L_s, sink=inp.sink)
    same = lambda G: float((_fp8_steps(G, O) == 0).mean())
    assert same(as_bf16) < 0.99
    assert same(as_fp32) >= 0.99


def test_the_rounding_helpers_are_what_they_claim():
    """hi is a truncation (never above p), hi + lo matches p to 2^-15, bf16 rounding is RNE."""
    e = np.exp(-np.linspace(0.0, 20.0, 4001))
    hl = _hi_lo_bf16(e)
    f = e.astype(np.float32).astype(np.float64)
    assert np.all(np.abs(hl - f) <= 2.0 ** -15 * f)
    hi = (e.astype(np.float32).view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32).astype(np.float64)
    assert np.all(hi <= f)
    ref = torch.from_numpy(e.astype(np.float32)).to(torch.bfloat16).double().numpy()
    assert np.array_equal(_single_bf16(e), ref)

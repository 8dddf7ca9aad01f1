"""Shared helpers of the GPU parity tests: run the C-ABI path, compare with the oracle.

Tolerances (stated once, used by every parity test):
  * O in fp32 output mode: for every (token, head) row,
        ||O_gpu - O_ref||_2 / ||O_ref||_2 <= 2e-3;
    a row whose reference is exactly 0 must be exactly 0 on the GPU.
  * LSE (log2): |LSE_gpu - LSE_ref| <= 1e-5; -inf must match exactly.
  * bf16 / e4m3 output ("compared after the same cast"), two rules, both applied:
      - interval: every GPU value lies between cast(O_ref - delta) and
        cast(O_ref + delta), delta = 2e-3 * rms(O_ref row);
      - code steps: every e4m3 code is within one step of the oracle's code
        e4m3(O_ref * inv_scale) on the number line (0x00 and 0x80 both count as 0);
        every bf16 value is within one ulp of bf16(O_ref), except where O_ref sits
        below the fp32 path's own error floor: there |O_gpu - O_ref| <= 2^-14 *
        rms(O_ref row) instead. (Where V cancels, O elements come arbitrarily close
        to 0 and one bf16 ulp shrinks with them; the fp32 accumulation and the
        2^-16 representation of P leave ~1e-6 absolute error, which no fp32 kernel
        removes. The dense FP8 path keeps P in f16 (2^-11), and its floor is
        2^-9 * rms(row): simulated on the oracle with only that rounding added, its
        worst element error is 2^-9.8 * rms. The e4m3 grid with inv_scale 64 bottoms
        out at 2^-15 in O units, above both floors, so its rule has no exception.)
  * amax: |amax_gpu - max|O_ref|| <= 2e-3 * max|O_ref|.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle.mla as om
from oracle import codecs
from split_kv_sparse_gb300 import binding as b

O_RTOL = 2e-3
LSE_ATOL = 1e-5

TORCH_OUT = {"f32": torch.float32, "bf16": torch.bfloat16, "e4m3": torch.uint8}


def check_status():
    st, site = b.mla_get_status()
    assert st == 0, f"device status {st:#x}, first timed-out wait site {site}"


def run_mla(inp, S: int, out_dtype: str = "f32", inv_scale: float = 1.0, with_amax: bool = False,
            keep_workspace: bool = False, num_sms: int = 0):
    """Whole decode step through mla_sparse_decode: S > 0 forces the (token,
    split) jobs (the direct path when S == 1); S == 0 takes the automatic plan;
    S == MLA_FORCE_BALANCED runs the balanced schedule where it applies. num_sms
    is the SM count the plan spreads the work over (0 = the device's)."""
    dev = torch.device("cuda")
    q, kv, idx = inp.q.to(dev), inp.kv.to(dev), inp.idx.to(dev)
    sink = inp.sink.to(dev) if inp.sink is not None else None
    plan = b.mla_decode_plan(inp.s_q, inp.topk, force_splits=S, num_sms=num_sms)
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=dev) if plan.workspace_bytes else None
    if ws is not None:
        b.mla_workspace_init(plan, ws)
    out = torch.empty(inp.s_q, 64, 512, dtype=TORCH_OUT[out_dtype], device=dev)
    lse = torch.empty(inp.s_q, 64, dtype=torch.float32, device=dev)
    amax = torch.empty(1, dtype=torch.float32, device=dev) if with_amax else None
    b.mla_sparse_decode(plan, inp.s_q, q, kv, inp.n_kv, idx, inp.sm_scale, sink, out_dtype, inv_scale, out,
                        lse, amax, ws)
    torch.cuda.synchronize()
    check_status()
    res = {"out": out.cpu(), "lse": lse.cpu().double().numpy(), "plan": plan}
    if with_amax:
        res["amax"] = float(amax.cpu()[0])
    if keep_workspace and ws is not None:
        res["o_acc"], res["lse_acc"] = workspace_views(plan, inp.s_q, ws)
    return res


def workspace_views(plan, s_q, ws):
    S = plan.num_splits
    o = ws[: S * s_q * 64 * 512 * 4].view(torch.float32).view(S, s_q, 64, 512)
    off = plan.lse_acc_offset
    l = ws[off: off + S * s_q * 64 * 4].view(torch.float32).view(S, s_q, 64)
    return o.cpu().double().numpy(), l.cpu().double().numpy()


def oracle_mla(inp):
    return om.attention(inp.q, inp.kv, inp.idx, inp.sm_scale, 512, sink=inp.sink)


def assert_o_close(O_gpu, O_ref, rtol=O_RTOL, what="O"):
    O_gpu = np.asarray(O_gpu, dtype=np.float64).reshape(-1, O_ref.shape[-1])
    O_ref = np.asarray(O_ref, dtype=np.float64).reshape(-1, O_ref.shape[-1])
    assert np.all(np.isfinite(O_gpu)), f"{what}: non-finite values"
    nref = np.linalg.norm(O_ref, axis=1)
    err = np.linalg.norm(O_gpu - O_ref, axis=1)
    zero = nref == 0
    assert np.all(O_gpu[zero] == 0), f"{what}: rows with a zero reference are not zero"
    rel = err[~zero] / nref[~zero]
    worst = float(rel.max()) if rel.size else 0.0
    assert worst <= rtol, f"{what}: worst row relative error {worst:.3e} > {rtol:.1e}"
    return worst


def assert_lse_close(L_gpu, L_ref, atol=LSE_ATOL, what="LSE"):
    L_gpu = np.asarray(L_gpu, dtype=np.float64)
    L_ref = np.asarray(L_ref, dtype=np.float64)
    ninf = np.isneginf(L_ref)
    assert np.array_equal(np.isneginf(L_gpu), ninf), f"{what}: -inf pattern differs"
    if (~ninf).any():
        worst = float(np.max(np.abs(L_gpu[~ninf] - L_ref[~ninf])))
        assert worst <= atol, f"{what}: worst abs error {worst:.3e} > {atol:.1e}"
        return worst
    return 0.0


def code_order_e4m3(codes) -> np.ndarray:
    """Position of each e4m3 code on the number line (sign-magnitude -> integer)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    mag = c & 0x7F
    return np.where((c >> 7) & 1, -mag, mag)


def code_order_bf16(bits) -> np.ndarray:
    """Position of each bf16 bit pattern on the number line (adjacent values differ by 1)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    mag = b & 0x7FFF
    return np.where((b >> 15) & 1, -mag, mag)


BF16_FLOOR = 2.0 ** -14          # sparse-MLA path: P as bf16 hi + lo (2^-16)
BF16_FLOOR_DENSE = 2.0 ** -9     # dense FP8 path: P as f16 (2^-11)


def assert_e4m3_within_one_step(gpu_codes: np.ndarray, O_ref: np.ndarray, inv_scale: float):
    """Every GPU e4m3 code is the oracle's code e4m3(O_ref * inv_scale) or a neighbour."""
    g = code_order_e4m3(np.asarray(gpu_codes, dtype=np.uint8).reshape(O_ref.shape))
    r = code_order_e4m3(codecs.e4m3_encode(O_ref * inv_scale))
    d = np.abs(g - r)
    assert d.max() <= 1, f"e4m3: {int((d > 1).sum())} codes more than one step from the oracle's (max {d.max()})"
    return float((d == 0).mean())


def assert_bf16_within_one_ulp(gpu_bits: np.ndarray, O_ref: np.ndarray, floor_rel: float = BF16_FLOOR):
    """Every GPU bf16 value is within one ulp of bf16(O_ref), or, below the path's own
    error floor, within floor_rel * rms(row) of O_ref."""
    gpu_bits = np.asarray(gpu_bits, dtype=np.uint16).reshape(O_ref.shape)
    d = np.abs(code_order_bf16(gpu_bits) - code_order_bf16(codecs.bf16_bits(O_ref)))
    floor = floor_rel * np.sqrt(np.mean(np.square(O_ref), axis=-1, keepdims=True))
    near = np.abs(codecs.bf16_decode(gpu_bits) - O_ref) <= floor
    bad = (d > 1) & ~near
    assert not bad.any(), f"bf16: {int(bad.sum())} values more than one ulp from bf16(O_ref) (max {d[bad].max()})"
    return float((d == 0).mean())


def _row_delta(O_ref, rtol):
    rms = np.sqrt(np.mean(np.square(O_ref), axis=-1, keepdims=True))
    return rtol * rms


def assert_cast_close(gpu_out: torch.Tensor, O_ref: np.ndarray, out_dtype: str, inv_scale: float = 1.0,
                      rtol: float = O_RTOL, bf16_floor: float = BF16_FLOOR):
    """Every GPU code lies between cast(O_ref - delta) and cast(O_ref + delta), and within one
    code step (e4m3) or one ulp (bf16) of the oracle's code; returns the fraction of codes
    identical to the oracle's."""
    delta = _row_delta(O_ref, rtol)
    if out_dtype == "bf16":
        g = gpu_out.float().double().numpy()
        lo = codecs.bf16_round(O_ref - delta)
        hi = codecs.bf16_round(O_ref + delta)
        same = assert_bf16_within_one_ulp(gpu_out.view(torch.int16).numpy().view(np.uint16), O_ref, bf16_floor)
    elif out_dtype == "e4m3":
        g = codecs.e4m3_decode(gpu_out.numpy())
        lo = codecs.e4m3_round((O_ref - delta) * inv_scale)
        hi = codecs.e4m3_round((O_ref + delta) * inv_scale)
        same = assert_e4m3_within_one_step(gpu_out.numpy(), O_ref, inv_scale)
    else:
        raise ValueError(out_dtype)
    ok = (g >= lo) & (g <= hi)
    assert ok.all(), f"{out_dtype}: {int((~ok).sum())} values outside the cast interval"
    return same
